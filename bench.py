#!/usr/bin/env python
"""Benchmark of one speculative-decoding selection step on GB300.

A step is one round: the exact top-k over the draft columns plus the fused
greedy verify over the target columns, issued as ONE spec_round launch.  The
default workload is 8 lanes x 7 drafts = 56 draft columns x V = 248,046 bf16
logits with k = 8, and a verify over 8 lanes x 8 target columns.

Prints one JSON line (rank 0).  ``value`` is logit GB/s (bytes of logits read
per round x rounds / time, all GPUs), ``us_per_round`` the time per round,
``roofline.frac`` the fraction of the measured HBM copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C2] [--impl ours|reference]

Timing: W untimed warm-up rounds, then exactly K rounds replayed as CUDA
graphs, bracketed by a barrier and a device synchronisation, timed with CUDA
events on the launching stream; max over ranks.  Every round reads a
different copy of the inputs from a ring larger than 4x the L2 cache, so
the logits come from HBM.  ``e2e`` repeats the metric through the host-buffer
entry point (spec_round_host): pinned host inputs copied in, outputs copied
back, every step.  ``cpu_baseline`` times the CPU oracle on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "µs per round and logit GB/s (% of GB300 HBM peak), top-k + greedy verify"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0      # GB300 HBM3e, the peak the targets are stated against
KERNEL_DIR = os.path.join(ROOT, "speculative_decoding_draft_column_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")

WORKLOADS = {
    "C1": "1 lane x 7 drafts: 7 draft columns x V=248,046 bf16 ~N(0,3) + 3 planted peaks, k=8; "
          "verify 1 lane x 8 target columns",
    "C2": "8 lanes x 7 drafts = 56 draft columns x V=248,046 bf16 ~N(0,3), k=8; verify 8 lanes x 8 target "
          "columns ~N(0,3) each with one planted strict maximum of 24.0 (its argmax), accepted length per lane "
          "uniform in 0..7",
    "C3": "1 lane, gamma 15: 15 draft columns x V=248,046 bf16 quantised to 64 levels (heavy ties), k=20; "
          "verify 3 lanes x 16 target columns",
    "C4": "64 lanes x 7 drafts = 448 draft columns x V=248,046 bf16, 90% N(0,2) / 10% one logit +12, k=20; "
          "verify 64 lanes x 8 target columns",
    "C5": "256 lanes x 15 drafts = 3,840 draft columns x V=248,046 bf16 ~N(0,3), k={k}; verify 256 lanes x 16 "
          "target columns",
    "C5s": "shortlist: 3,840 draft columns x 131,072 bf16 ~N(0,3) whose local ids map to vocabulary ids through "
           "a seeded 131,072-entry id map (spec_topk_mapped), k={k}; no verify",
}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100_000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--config", default="C2", choices=sorted(WORKLOADS))
    p.add_argument("--k", type=int, default=None, help="k for C5 and C5s (1, 8, 20 or 64)")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--part", default="round", choices=["round", "split", "topk", "verify"],
                   help="round: spec_round, one fused launch (default); split: spec_topk then spec_verify_v, two "
                        "launches a round; topk / verify: that call alone on its own columns")
    p.add_argument("--kernel", default="auto", choices=["auto", "warp", "cta", "gm"],
                   help="streaming kernel (spec_set_kernel); auto picks by round size")
    p.add_argument("--sampled", action="store_true",
                   help="verify by speculative sampling (T 1.0, top_p 0.95, top_k 20, one-hot drafts; "
                        "spec_round_sampled) instead of greedy; measures the kernel line only (no e2e, no CPU arm)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--head", type=int, default=0, metavar="N",
                   help="instead of a round: N hidden states through the full Q4 shortlist head "
                        "(131,072 x 5,120, 356.5 MB) and the mapped top-k (k=8), spec_shortlist_topk")
    p.add_argument("--no-also", action="store_true",
                   help="skip the extra kernel timings of C1 and C4 that the default C2 run reports under 'also'")
    return p.parse_args(argv)


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        if v > 0:
            return v, "of measured"
    except Exception:
        pass
    return FALLBACK_HBM_GBS, "of fallback"


def source_hash() -> str:
    """sha256 (first 16 hex digits) over the kernel sources, in name order."""
    h = hashlib.sha256()
    for name in sorted(os.listdir(KERNEL_DIR)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(KERNEL_DIR, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


# The bench names the kernel that ran, as the library reports it
# (spec_last_kernel: the kernel of the calling thread's last round launch).
KERNEL_NAMES = {1: "wrp::spec_round_kernel", 2: "cta::spec_round_kernel", 3: "gm::spec_round_kernel"}
KERNEL_CHOICES = {"auto": 0, "warp": 1, "cta": 2, "gm": 3}


def kernel_name(sd) -> str:
    return KERNEL_NAMES.get(sd.spec_last_kernel(), "unknown")


def recorded_traffic(config: str):
    """DRAM bytes per launch from a committed ncu capture, if the kernel
    source has not changed since it was taken (else None)."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        e = t.get(config)
        if e and e.get("source_sha256_16") == source_hash():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def make_workload(config: str, k: int | None, seed_offset: int = 0):
    import synth
    fn = synth.CONFIGS[config]
    kw = {}
    if config in ("C5", "C5s") and k is not None:
        kw["k"] = k
    if seed_offset:
        import inspect
        kw["seed"] = inspect.signature(fn).parameters["seed"].default + 1000 * seed_offset
    return fn(**kw)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 9:
                    rows.append(p)
        os.unlink(self.path)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# multi-process plumbing (one process per GPU; replicas, no data exchange)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return world, rank, local


def dist_init(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value over all ranks (plain max when there is one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------------------
# the CPU oracle (baseline / reference arm)
# ---------------------------------------------------------------------------

def oracle_round(r, threads: int, cols=None, n: int | None = None):
    """The oracle over a round (or over columns `cols` cut to their first n
    elements); returns the logit bytes it read."""
    import oracle
    if cols is None:
        if r.id_map is not None:
            oracle.topk_mapped(r.draft, r.k, r.id_map, threads=threads)
        else:
            oracle.topk(r.draft, r.k, threads=threads)
        if r.target is not None:
            oracle.verify(r.target, r.drafts, threads=threads)
        return r.logit_bytes()
    dc, tc = cols
    nb = 0
    if len(dc):
        x = r.draft[dc, :n]
        if r.id_map is not None:
            oracle.topk_mapped(x, min(r.k, x.shape[1]), r.id_map[:x.shape[1]], threads=threads)
        else:
            oracle.topk(x, min(r.k, x.shape[1]), threads=threads)
        nb += x.size * 2
    if len(tc):
        t = r.target[tc, :n]
        oracle.argmax(t, threads=threads)
        nb += t.size * 2
    return nb


def _time_oracle_rounds(r, threads: int, budget_s: float):
    t0 = time.perf_counter()
    rounds, nbytes = 0, 0
    while True:
        nbytes += oracle_round(r, threads)
        rounds += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return rounds, nbytes, time.perf_counter() - t0


def cpu_baseline(r, budget_s: float = 3.0, one_core_max_bytes: int = 100_000_000):
    """The oracle over whole rounds on every host core (and, for rounds of
    at most `one_core_max_bytes` of logits, on one core)."""
    threads = os.cpu_count() or 1
    oracle_round(r, threads)                 # warm (page in, build)
    rounds, nbytes, dt = _time_oracle_rounds(r, threads, budget_s)
    ncols = r.cols + (0 if r.target is None else r.target.shape[0])
    out = {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
           "sample": f"{rounds} full rounds of the same workload ({r.cols} top-k columns + "
                     f"{0 if r.target is None else r.target.shape[0]} verify columns each), "
                     f"{dt:.2f} s wall on {threads} threads",
           "us_per_round": round(dt / rounds * 1e6, 1), "columns_per_s": round(rounds * ncols / dt, 1)}
    if r.logit_bytes() <= one_core_max_bytes:
        r1, b1, d1 = _time_oracle_rounds(r, 1, 0.0)        # one round on one thread
        out["one_core"] = {"value": round(b1 / d1 / 1e9, 4), "unit": "GB/s", "us_per_round": round(d1 / r1 * 1e6, 1),
                           "columns_per_s": round(r1 * ncols / d1, 1)}
    return out


def run_reference(args):
    """The oracle as the reference arm, on the host cores.  A step is one whole
    round of the workload (every draft and target column) when W + K whole
    rounds fit in about two minutes (C1-C4); otherwise a bounded sample of it
    (C5): the first n logits of one column per host thread."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    r = make_workload(args.config, args.k)
    threads = os.cpu_count() or 1
    nt = 0 if r.target is None else r.target.shape[0]
    budget_s = 120.0
    t0 = time.perf_counter()
    oracle_round(r, threads)                                   # the first warm-up step
    t_round = time.perf_counter() - t0
    whole = (args.steps + args.warmup) * t_round <= budget_s
    if whole:
        def step(i):
            return oracle_round(r, threads)
        sample = (f"each step: one whole round ({r.cols} top-k columns" + (f" + {nt} verify columns" if nt else "")
                  + f") on {threads} threads")
        cores = threads
    else:
        m = min(threads, r.cols, nt) if nt else min(threads, r.cols)
        b = oracle_round(r, threads, cols=(list(range(m)), list(range(m)) if nt else []), n=r.V)
        per_byte = t_round / r.logit_bytes()
        n_elems = max(64, min(r.V, int(budget_s / max(1, args.steps + args.warmup) / per_byte / b * r.V)))

        def step(i):
            dc = [(i * m + j) % r.cols for j in range(m)]
            tc = [(i * m + j) % nt for j in range(m)] if nt else []
            return oracle_round(r, threads, cols=(dc, tc), n=n_elems)
        sample = (f"each step: the oracle's top-k over the first {n_elems} logits of {m} draft columns"
                  + (f" and its argmax over the first {n_elems} logits of {m} target columns" if nt else "")
                  + f", one column per thread ({m} threads); a whole round takes {t_round:.1f} s")
        cores = m

    for i in range(max(0, args.warmup - 1)):
        step(i)
    t0 = time.perf_counter()
    nbytes = 0
    for i in range(args.steps):
        nbytes += step(i)
    dt = time.perf_counter() - t0
    gbs = nbytes / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(args, r, None),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    if whole:
        line["us_per_round"] = round(dt / args.steps * 1e6, 1)
    print(json.dumps(line), flush=True)
    return 0


def input_hashes(r) -> dict:
    """sha256[:16] of every input buffer of the round (seeded, so fixed per
    workload and seed)."""
    import synth
    bufs = (("draft_logits", r.draft), ("target_logits", r.target), ("drafts", r.drafts), ("id_map", r.id_map))
    return {name: synth.content_hash(a) for name, a in bufs if a is not None}


def workload_config(args, r, ring):
    desc = WORKLOADS[args.config].format(k=r.k)
    c = {"workload": f"{args.config}: {desc}", "cols": r.cols, "V": r.V, "k": r.k, "lanes": r.lanes,
         "gamma": r.gamma, "bytes_per_round": r.logit_bytes(), "parallelism": "replicas (one independent round "
         "per GPU, no data exchange)", "input_sha256_16": input_hashes(r)}
    if ring is not None:
        c["l2"] = (f"inputs rotated through a ring of {ring[0]} copies ({ring[1] / 1e6:.0f} MB, > 4x the "
                   f"{ring[2] / 1e6:.0f} MB L2): every round reads its logits from HBM")
        c["launch"] = ("spec_round_sampled" if args.sampled else "spec_topk_mapped" if r.id_map is not None
                       else "spec_round") + ": one kernel per round; K rounds replayed as CUDA graphs"
    if args.sampled:
        c["verify"] = "sampled: T 1.0, top_p 0.95, top_k 20, one-hot drafts, seeded uniforms"
    part = getattr(args, "part", "round")
    if part != "round":
        c["part"] = {"split": "spec_topk then spec_verify_v: two launches a round",
                     "topk": "spec_topk alone on the draft columns (value = their logit GB/s)",
                     "verify": "spec_verify_v alone on the target columns (value = their logit GB/s)"}[part]
    return c


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def replay_us(one, K: int, R: int, stream, sd) -> float:
    """Mean µs per call of one(i), i = 0..K-1, replayed as CUDA graphs of up
    to ~1000 calls (inputs rotating through R copies), timed with CUDA events
    on `stream` after one untimed replay."""
    import torch
    chunk = min(K, R * max(1, 1000 // R))
    n_full, rem = divmod(K, chunk)
    graphs = []
    for n in ([chunk] + ([rem] if rem else [])):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                one(i)
        graphs.append(g)
    with torch.cuda.stream(stream):
        graphs[0].replay()
    stream.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n_full):
            graphs[0].replay()
        if rem:
            graphs[1].replay()
        e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1) * 1e3 / K


def also_rounds(dev, stream, sd, peak: float, clocks) -> dict:
    """The other two workloads the targets name, timed on the same replay
    loop as the headline: C1 (7 + 8 columns; the bar is 3x its
    bytes/bandwidth floor) and C4 (448 + 512 columns; the bar is 60% of HBM
    peak), one spec_round per round, inputs rotating through > 4x L2."""
    import numpy as np
    import torch
    out = {}
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    clocks.start()
    for name, K in (("C1", 2000), ("C4", 200)):
        r = make_workload(name, None)
        R = max(2, math.ceil(4 * l2 / r.logit_bytes()))
        xs = [torch.from_numpy(r.draft.view(np.int16)).to(dev) for _ in range(R)]
        ts = [torch.from_numpy(r.target.view(np.int16)).to(dev) for _ in range(R)]
        d = torch.from_numpy(r.drafts).to(dev)
        vals = torch.empty((r.cols, r.k), dtype=torch.int16, device=dev)
        ids = torch.empty((r.cols, r.k), dtype=torch.int32, device=dev)
        acc = torch.empty(r.lanes, dtype=torch.int32, device=dev)
        com = torch.empty((r.lanes, r.gamma + 1), dtype=torch.int32, device=dev)
        sd.spec_reserve(r.cols, r.k, r.lanes, r.gamma)

        def one(i):
            sd.spec_round(xs[i % R], r.cols, r.V, r.k, vals, ids, ts[i % R], d, r.lanes, r.gamma, acc, com)

        with torch.cuda.stream(stream):
            for i in range(5):
                one(i)
        stream.synchronize()
        kname = kernel_name(sd)
        us = replay_us(one, K, R, stream, sd)
        b = r.logit_bytes()
        floor_meas, floor_nom = b / (peak * 1e3), b / (NOMINAL_HBM_GBS * 1e3)
        out[name] = {"workload": f"{name}: " + WORKLOADS[name].format(k=r.k), "bytes_per_round": b,
                     "us_per_round": round(us, 3), "gb_s": round(b / us / 1e3, 1),
                     "frac_of_measured_hbm": round(b / us / 1e3 / peak, 4),
                     "frac_of_nominal_hbm": round(b / us / 1e3 / NOMINAL_HBM_GBS, 4),
                     "floor_us_measured_hbm": round(floor_meas, 3), "floor_multiple_measured": round(us / floor_meas, 2),
                     "floor_us_nominal_hbm": round(floor_nom, 3), "floor_multiple_nominal": round(us / floor_nom, 2),
                     "rounds": K, "kernel": kname}
        del xs, ts
        torch.cuda.empty_cache()
    out["clocks"] = clocks.stop()
    out["timing"] = "as the headline: CUDA events around K graph-replayed spec_round launches, inputs from HBM"
    return out


def run_ours(args):
    import numpy as np
    import torch

    world, rank, local = dist_env()
    assert torch.cuda.is_available(), "bench.py needs a CUDA device (there is no CPU fallback)"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    import speculative_decoding_draft_column_gb300 as sd

    r = make_workload(args.config, args.k, seed_offset=rank)   # independent lanes per GPU
    if args.sampled and r.id_map is not None:
        raise SystemExit("--sampled needs target columns; the shortlist workload has none")
    if args.part != "round" and (args.sampled or r.id_map is not None or not r.lanes):
        raise SystemExit("--part other than round needs a greedy round with draft and target columns")
    cols, V, k, lanes, gamma = r.cols, r.V, r.k, r.lanes, max(r.gamma, 1)
    bytes_round = r.logit_bytes()
    # logits read per step, and per launch of the call(s) timed
    bytes_step = {"round": bytes_round, "split": bytes_round, "topk": r.draft.nbytes,
                  "verify": 0 if r.target is None else r.target.nbytes}[args.part]
    per_step = 2 if args.part == "split" else 1
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    R = max(2, math.ceil(4 * l2 / bytes_round))
    xs = [torch.from_numpy(r.draft.view(np.int16)).to(dev) for _ in range(R)]
    ts = [torch.from_numpy(r.target.view(np.int16)).to(dev) if lanes else None for _ in range(R)]
    drafts = torch.from_numpy(r.drafts).to(dev) if lanes else None
    id_map = torch.from_numpy(r.id_map).to(dev) if r.id_map is not None else None
    vals = torch.empty((cols, k), dtype=torch.int16, device=dev)
    ids = torch.empty((cols, k), dtype=torch.int32, device=dev)
    acc = torch.empty(max(lanes, 1), dtype=torch.int32, device=dev)
    com = torch.empty((max(lanes, 1), gamma + 1), dtype=torch.int32, device=dev)
    sd.spec_set_kernel(KERNEL_CHOICES[args.kernel])
    sd.spec_reserve(cols, k, lanes, gamma)
    stream = torch.cuda.Stream(device=dev)

    if args.sampled:
        uni = torch.from_numpy(np.random.default_rng(12345 + rank).random((max(lanes, 1), gamma + 1, 2))).to(dev)

        def one(i):
            sd.spec_round_sampled(xs[i % R], cols, V, k, vals, ids, ts[i % R], drafts, lanes, gamma,
                                  1.0, 0.95, 20, uni, acc, com)
    elif id_map is not None:
        def one(i):
            sd.spec_topk_mapped(xs[i % R], cols, V, k, id_map, vals, ids)
    elif args.part == "split":
        def one(i):
            sd.spec_topk(xs[i % R], cols, V, k, vals, ids)
            sd.spec_verify_v(ts[i % R], drafts, lanes, gamma, V, acc, com)
    elif args.part == "topk":
        def one(i):
            sd.spec_topk(xs[i % R], cols, V, k, vals, ids)
    elif args.part == "verify":
        def one(i):
            sd.spec_verify_v(ts[i % R], drafts, lanes, gamma, V, acc, com)
    else:
        def one(i):
            sd.spec_round(xs[i % R], cols, V, k, vals, ids, ts[i % R], drafts, lanes, gamma, acc, com)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            one(i)
        if args.part == "split":
            sd.spec_topk(xs[0], cols, V, k, vals, ids)
            kname = kernel_name(sd)
            sd.spec_verify_v(ts[0], drafts, lanes, gamma, V, acc, com)
            kname += " + " + kernel_name(sd)
        else:
            kname = kernel_name(sd)
    stream.synchronize()

    K = args.steps
    chunk = min(K, R * max(1, 1000 // R))
    n_full, rem = divmod(K, chunk)
    graphs = []
    c0 = sd.spec_launch_count()
    for n in ([chunk] + ([rem] if rem else [])):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                one(i)
        graphs.append(g)
    captured = sd.spec_launch_count() - c0
    assert captured == (chunk + rem) * per_step
    with torch.cuda.stream(stream):
        graphs[0].replay()                   # untimed: upload / warm the graph
    stream.synchronize()

    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None else str(local))
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    clocks.start()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n_full):
            graphs[0].replay()
        if rem:
            graphs[1].replay()
        e1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    barrier(world, dev)
    ms = e0.elapsed_time(e1)
    also = None
    if (world == 1 and not args.no_also and args.config == "C2" and args.part == "round" and not args.sampled
            and args.kernel == "auto"):
        also = also_rounds(dev, stream, sd, hbm_peak()[0], ClockSampler(f"GPU-{uuid}" if uuid is not None else str(local)))
    ms_max = max_over_ranks(ms, world, dev)
    launches = (n_full * chunk + rem) * per_step

    # end to end through the host-buffer entry point
    e2e = None
    if not args.no_e2e and not args.sampled and args.part == "round":
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
        hd = pin(r.draft.view(np.int16))
        ht = pin(r.target.view(np.int16)) if lanes else None
        hdr = pin(r.drafts) if lanes else None
        hv = torch.empty((cols, k), dtype=torch.int16).pin_memory()
        hi = torch.empty((cols, k), dtype=torch.int32).pin_memory()
        ha = torch.empty(max(lanes, 1), dtype=torch.int32).pin_memory()
        hc = torch.empty((max(lanes, 1), gamma + 1), dtype=torch.int32).pin_memory()
        sd.spec_set_stream(stream)
        api = "spec_round_host (pinned host buffers; H2D, kernel, D2H, stream sync per step)"

        def host_step():
            sd.lib.spec_round_host(hd.data_ptr(), cols, V, k, hv.data_ptr(), hi.data_ptr(),
                                   ht.data_ptr() if lanes else None, hdr.data_ptr() if lanes else None, lanes,
                                   gamma, ha.data_ptr() if lanes else None, hc.data_ptr() if lanes else None)

        if id_map is not None:
            # the shortlist has no host-buffer entry point: the caller's own
            # copies around spec_topk_mapped (the map stays on the device)
            api = ("torch copies from pinned host buffers on the library stream + spec_topk_mapped + "
                   "copies back, stream sync per step")
            xd = xs[0]

            def host_step():
                with torch.cuda.stream(stream):
                    xd.copy_(hd, non_blocking=True)
                    sd.spec_topk_mapped(xd, cols, V, k, id_map, vals, ids)
                    hv.copy_(vals, non_blocking=True)
                    hi.copy_(ids, non_blocking=True)
                stream.synchronize()

        for _ in range(5):
            host_step()
        n_e2e = max(20, min(K, 300))
        barrier(world, dev)
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            host_step()
        dt = max_over_ranks(time.perf_counter() - t0, world, dev)
        if sd.spec_last_error():
            raise RuntimeError(sd.spec_last_error())
        h2d = r.draft.nbytes + (r.target.nbytes + r.drafts.nbytes if lanes else 0)
        d2h = vals.numel() * 2 + ids.numel() * 4 + (acc.numel() * 4 + com.numel() * 4 if lanes else 0)
        e2e = {"value": round(world * bytes_round * n_e2e / dt / 1e9, 2), "unit": "GB/s",
               "us_per_round": round(dt / n_e2e * 1e6, 2), "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": n_e2e,
               "api": api}

    if rank != 0:
        return 0
    peak, peak_src = hbm_peak()
    us_round = ms_max * 1e3 / K
    gbs = world * bytes_step * K / (ms_max * 1e-3) / 1e9
    per_launch_us = ms * 1e3 / launches
    # the roofline of one launch; for the split round, of one step (two launches)
    unit_us = per_launch_us * per_step
    achieved = bytes_step / (unit_us * 1e-6) / 1e9
    line = {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_max / K, 6), "us_per_round": round(us_round, 3),
        "pct_of_hbm_peak": round(100 * gbs / world / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_hbm": round(100 * gbs / world / peak, 2),
        "hbm_peaks_gbs": {"nominal": NOMINAL_HBM_GBS, "measured_copy": peak},
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; see synth/)",
        "config": workload_config(args, r, (R, R * bytes_round, l2)),
        "roofline": {"bound": "hbm", "kernel": kname,
                     "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_source": peak_src,
                     "traffic": recorded_traffic(args.config) if args.part == "round" and not args.sampled
                     and args.kernel == "auto" else None,
                     "algorithmic_bytes_per_launch": bytes_step if per_step == 1 else None,
                     "launch_us": round(per_launch_us, 3),
                     "timing": "CUDA events around K graph-replayed launches on the launching stream; "
                               "per-launch time includes the graph's inter-launch gap"},
        "gpu_launches": int(launches),
        "clocks": clk,
    }
    if e2e:
        line["e2e"] = e2e
    if also:
        line["also"] = also
    if world == 1 and not args.no_cpu_baseline and not args.sampled and args.part == "round":
        line["cpu_baseline"] = cpu_baseline(r)
    print(json.dumps(line), flush=True)
    return 0


def run_head(args):
    """The Q4 shortlist head workload: N hidden states (5,120 wide, N(0,1))
    through the full head (131,072 rows, 356.5 MB of packed weights and
    scales, larger than L2, so every call streams it from HBM) into logits,
    then the mapped top-k (k = 8).  One spec_shortlist_topk per step."""
    import numpy as np
    import torch
    import synth
    import speculative_decoding_draft_column_gb300 as sd
    world, rank, local = dist_env()
    assert torch.cuda.is_available(), "bench.py needs a CUDA device (there is no CPU fallback)"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cols, k = args.head, 8
    rows, d = synth.SHORTLIST, synth.HIDDEN
    wq, sc = synth.q4_head(41 + rank)
    h = synth.hidden_states(42 + rank, cols, d)
    id_map = synth.shortlist_map(43)
    w = torch.from_numpy(wq).to(dev)
    s = torch.from_numpy(sc.view(np.int16)).to(dev)
    wp, sp = torch.empty_like(w), torch.empty_like(s)
    sd.spec_shortlist_pack(w, s, rows, d, wp, sp)
    del w, s
    hd = torch.from_numpy(h.view(np.int16)).to(dev)
    m = torch.from_numpy(id_map).to(dev)
    lg = torch.empty((cols, rows), dtype=torch.int16, device=dev)
    vals = torch.empty((cols, k), dtype=torch.int16, device=dev)
    ids = torch.empty((cols, k), dtype=torch.int32, device=dev)
    sd.spec_reserve(cols, k, 0, 1)
    stream = torch.cuda.Stream(device=dev)

    def one(i):
        sd.spec_shortlist_topk(hd, cols, d, wp, sp, rows, m, k, lg, vals, ids)

    def logits_only(i):
        sd.spec_shortlist_logits(hd, cols, d, wp, sp, rows, lg)

    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            one(i)
    stream.synchronize()
    K = args.steps
    uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None else str(local))
    clocks.start()
    us = replay_us(one, K, 1, stream, sd)
    us_logits = replay_us(logits_only, K, 1, stream, sd)
    clk = clocks.stop()
    head_bytes = wq.nbytes + sc.nbytes
    passes = -(-cols // 16)
    peak, peak_src = hbm_peak()
    tflops = 2.0 * rows * d * cols / (us_logits * 1e-6) / 1e12
    line = {
        "metric": "µs per call and head GB/s, Q4 shortlist head logits + mapped top-k", "value": round(us, 3),
        "unit": "µs", "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 6),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16 x int4 -> fp32",
        "data": "synthetic (seeded; see synth/)",
        "config": {"workload": f"{cols} hidden states x 5,120 (bf16 N(0,1)) through the Q4 shortlist head "
                               f"(131,072 rows; 4-bit weights, fp16 scale per 64; 356.5 MB), mapped top-k k={k}",
                   "l2": "the head (356.5 MB) exceeds the L2: every call streams it from HBM",
                   "launch": f"spec_shortlist_topk: {passes} logits launch(es) of up to 16 hidden states, "
                             "then one spec_topk_mapped launch; K calls replayed as CUDA graphs"},
        "us_logits": round(us_logits, 3), "us_topk": round(us - us_logits, 3),
        "roofline": {"bound": "hbm", "kernel": "q4::logits_kernel",
                     "achieved": round(head_bytes * passes / (us_logits * 1e-6) / 1e9, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(head_bytes * passes / (us_logits * 1e-6) / 1e9 / peak, 4),
                     "peak_source": peak_src, "traffic": None,
                     "algorithmic_bytes_per_launch": head_bytes,
                     "head_passes_per_call": passes, "tensor_tflops": round(tflops, 1)},
        "gpu_launches": int(K * (passes + 1)),
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.head:
        return run_head(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
