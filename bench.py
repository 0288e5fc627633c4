"""Throughput of speculative-sampling verification on GB300.

One step = one chain verification of a batch of B = 256 sequences with
gamma = 7 drafts over a V = 128256 bf16 vocabulary (2048 target rows + 1792
draft rows, 985,006,080 bytes of logits): every stage of the path (policy and
softmax statistics, acceptance, residual and bonus draws) runs inside the
timed call.  Inputs are resident in HBM and larger than L2, so every step
streams them from DRAM.  Metric: verified vocabulary rows per second,
B * (gamma + 1) per step.

Arms:
  default           the CUDA library through its Python binding
  --impl reference  the CPU oracle (the plain float64 restatement of the
                    method) on this host's cores, on a bounded sample

--op filters times the same chain verification with top-p 0.9 and min-p 0.05
on both sides of every sequence (same metric);
--op overlap times the per-position overlap beta_i = sum min(p_i, q_i) of
the same workload instead (metric: positions per second, B * gamma per step);
--op typical times typical acceptance (epsilon 0.0625, delta 0.5; metric:
target rows per second, B * (gamma + 1) per step); --op rerank times the
EAGLE-2 rerank of 256 draft trees of 1024 nodes (top 64; metric: trees per
second).

Under torchrun each rank verifies its own batch on its own GPU (weak
scaling, no collective on the data path); rank 0 prints one JSON line.
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = 2
METRIC = "verified vocab rows/s (B*(gamma+1))"
CSRC = os.path.join(ROOT, "speculative_decoding_verification_temp_gb300", "csrc")
# the ncu summary of the dominant kernel on this workload (the rows kernel of
# the chain path): its DRAM traffic per launch, valid while the kernel's
# sources hash to the recorded value
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "chain_rows_kernel_b256_g7_v128256_bf16.md")
TRAFFIC_UNIT = "chain_rows.cu"
# kernels the library launches per chain call on this workload: rows, decide,
# weights, search, precise jobs, precise search
LAUNCHES_PER_STEP = 3  # rows kernel, draw kernel, precise kernel
# --op filters: top-p and min-p of every sequence (both sides); the rows,
# filter, draw and precise kernels run
FILTER_TOP_P, FILTER_MIN_P = 0.9, 0.05
FILTER_LAUNCHES_PER_STEP = 4
OVERLAP_METRIC = "overlap positions/s (B*gamma)"
L2_BYTES = 129e6
OVERLAP_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "overlap_kernel_b256_g7_v128256_bf16.md")
TYPICAL_METRIC = "typical-acceptance target rows/s (B*(gamma+1))"
TYPICAL_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "typical_rows_b256_g7_v128256_bf16.md")
TYPICAL_EPS, TYPICAL_DELTA = 0.0625, 0.5


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, world, dev):
    """The largest of the ranks' values of x (a float); x itself on one rank."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, rows_per_rank_step, steps, seconds):
    """Whole-job throughput: the rows every rank verified over the slowest rank's time."""
    return world * rows_per_rank_step * steps / seconds


def kernel_source_hash(unit=TRAFFIC_UNIT):
    """Hash of a kernel's sources: its translation unit (which also holds its
    launch function) and the local headers it includes, transitively."""
    seen, todo = set(), [unit]
    while todo:
        name = todo.pop()
        if name in seen:
            continue
        seen.add(name)
        with open(os.path.join(CSRC, name), encoding="utf-8") as f:
            for line in f:
                line = line.strip()
                if line.startswith('#include "'):
                    inc = line.split('"')[1]
                    if os.path.exists(os.path.join(CSRC, inc)):
                        todo.append(inc)
    h = hashlib.sha256()
    for name in sorted(seen):
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def recorded_traffic(path=TRAFFIC_FILE, unit=TRAFFIC_UNIT):
    """Per-launch DRAM bytes from the committed ncu summary, if the kernel is unchanged.

    The summary holds lines "- source_hash: H" and "- dram_bytes_per_launch: N".
    """
    rec = {}
    try:
        with open(path) as f:
            for line in f:
                line = line.strip()
                if line.startswith("- ") and ":" in line:
                    key, val = line[2:].split(":", 1)
                    rec[key.strip()] = val.strip()
    except OSError:
        return None
    if rec.get("source_hash") != kernel_source_hash(unit):
        return None
    try:
        return int(rec["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                self.out = ""

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def clocks_of(clk, gpu_index, call):
    """The clocks sampled during a timed region, or, when it was too short for
    three samples of the 100 ms sampler, those of a 1.5 s window of
    back-to-back calls right after it."""
    import torch
    clocks = clk.summary()
    if clocks["samples"] >= 3:
        return clocks
    with ClockSampler(gpu_index) as clk2:
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < 1.5:
            for _ in range(50):
                call()
            torch.cuda.synchronize()
    clocks = clk2.summary()
    clocks["window"] = "1.5 s of back-to-back calls right after the timed region"
    return clocks


def oracle_sample_rate(w, n_seqs, min_s=0.0, max_passes=1):
    """The CPU oracle on the first n_seqs sequences, repeated until min_s seconds
    (at most max_passes passes): (verified rows per second, seconds, passes).
    w["filters"], when present, holds the top-p / min-p arrays of the call."""
    from oracle import verify as ov
    gamma = w["gamma"]
    t0 = time.perf_counter()
    passes = 0
    while True:
        ov.verify_chain(w["target"], w["draft"], w["tokens"], w["target_temperature"],
                        w["draft_temperature"], w["target_top_k"], w["draft_top_k"],
                        seed=w["seed"], seqs=range(n_seqs), **w.get("filters", {}))
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_s or passes >= max_passes:
            break
    return passes * n_seqs * (gamma + 1) / dt, dt, passes


def _oracle_worker(spec, seqs, passes=1):
    """One process of the all-core CPU baseline: the oracle on `seqs`, `passes`
    times, the workload's arrays attached from shared memory."""
    from multiprocessing import shared_memory
    sys.path.insert(0, ROOT)
    from oracle import verify as ov
    shms, arrs = [], {}
    for key, (name, shape, dtype) in spec["arrays"].items():
        shm = shared_memory.SharedMemory(name=name)
        shms.append(shm)
        arrs[key] = np.ndarray(shape, dtype=dtype, buffer=shm.buf)
    t0 = time.perf_counter()
    for _ in range(passes):
        ov.verify_chain(arrs["target"], arrs["draft"], arrs["tokens"], arrs["tt"], arrs["td"],
                        None, None, seed=spec["seed"], seqs=seqs, **spec["filters"])
    dt = time.perf_counter() - t0
    del arrs
    for shm in shms:
        shm.close()
    return dt


def oracle_all_cores(w, n_seqs, min_s=0.0):
    """The CPU oracle on the first n_seqs sequences, split over every host core
    (spawned processes reading the workload from shared memory), repeated so
    that the timed run takes about min_s seconds: (rows per second, wall
    seconds, processes, passes)."""
    import concurrent.futures as cf
    import multiprocessing as mp
    from multiprocessing import shared_memory
    cores = os.cpu_count() or 1
    arrays = {"target": w["target"], "draft": w["draft"], "tokens": w["tokens"],
              "tt": np.asarray(w["target_temperature"], np.float32),
              "td": np.asarray(w["draft_temperature"], np.float32)}
    shms, spec = [], {"arrays": {}, "seed": w["seed"], "filters": w.get("filters", {})}
    try:
        for key, a in arrays.items():
            a = np.ascontiguousarray(a)
            shm = shared_memory.SharedMemory(create=True, size=max(1, a.nbytes))
            shms.append(shm)
            np.ndarray(a.shape, dtype=a.dtype, buffer=shm.buf)[...] = a
            spec["arrays"][key] = (shm.name, a.shape, a.dtype.str)
        parts = [list(range(i, n_seqs, cores)) for i in range(cores)]
        parts = [p for p in parts if p]
        with cf.ProcessPoolExecutor(len(parts), mp_context=mp.get_context("spawn")) as ex:
            # start-up outside the timing; one pass sizes the repeat count
            list(ex.map(_oracle_worker, [spec] * len(parts), [[p[0]] for p in parts]))
            t0 = time.perf_counter()
            list(ex.map(_oracle_worker, [spec] * len(parts), parts))
            one = time.perf_counter() - t0
            passes = max(1, min(50, int(min_s / max(one, 1e-6))))
            t0 = time.perf_counter()
            list(ex.map(_oracle_worker, [spec] * len(parts), parts, [passes] * len(parts)))
            dt = time.perf_counter() - t0
    finally:
        for shm in shms:
            shm.close()
            shm.unlink()
    return passes * n_seqs * (w["gamma"] + 1) / dt, dt, len(parts), passes


def config_entry(w):
    filt = ", top-p 0.9 and min-p 0.05 on both sides" if w.get("filters") else ""
    return {"workload": f"chain verify B={w['B']} gamma={w['gamma']} V={w['V']} {w['dtype']} "
                        f"(temperature 1, Zipf logits, draft sigma 0.4{filt})",
            "B": w["B"], "gamma": w["gamma"], "V": w["V"],
            "logit_bytes_per_step": logit_bytes(w),
            "l2": l2_note(logit_bytes(w), "logits")}


def l2_note(nbytes, what):
    side = "larger" if nbytes > L2_BYTES else "smaller"
    return f"inputs {side} than L2 ({nbytes / 1e6:.0f} MB of {what} per step)"


def logit_bytes(w):
    esize = 2 if w["dtype"] == "bf16" else 4
    return (w["B"] * (w["gamma"] + 1) + w["B"] * w["gamma"]) * w["V"] * esize


def bench_workload(args):
    """The timed workload: B = 256, gamma = 7, V = 128256 bf16, or the same
    recipe with --batch sequences (smaller cases for profiling).  --op filters
    adds top-p 0.9 and min-p 0.05 on both sides of every sequence."""
    from speculative_decoding_verification_temp_gb300 import workloads
    if not args.batch:
        w = workloads.config(WORKLOAD)
    else:
        c = dict(workloads.CONFIGS[WORKLOAD])
        c.pop("kind")
        c["B"] = args.batch
        w = workloads.make_chain(seed=1000 + WORKLOAD, **c)
    if getattr(args, "op", "verify") == "filters":
        P = np.full(w["B"], FILTER_TOP_P, np.float32)
        M = np.full(w["B"], FILTER_MIN_P, np.float32)
        w["filters"] = dict(target_top_p=P, draft_top_p=P, target_min_p=M, draft_min_p=M)
    return w


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from speculative_decoding_verification_temp_gb300 import workloads
    w = bench_workload(args)
    # a bounded sample per step: about a minute of oracle work in all at the
    # default step count (about 8 ms per sequence on one core)
    n_seqs = max(1, min(args.reference_seqs, 7500 // max(1, args.steps)))
    rows_per_step = n_seqs * (w["gamma"] + 1)
    for _ in range(args.warmup):
        oracle_sample_rate(w, min(n_seqs, 4))  # (rate, seconds, passes)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample_rate(w, n_seqs)
    dt = time.perf_counter() - t0
    value = rows_per_step * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config_entry(w),
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": 1, "kind": "oracle",
                         "sample": f"first {n_seqs} of {w['B']} sequences per step"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    import torch.distributed as dist

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_verification_temp_gb300 as sv
    from speculative_decoding_verification_temp_gb300 import workloads

    w = bench_workload(args)
    B, gamma, V = w["B"], w["gamma"], w["V"]
    seed = w["seed"] + rank  # each rank verifies its own batch
    rows = B * (gamma + 1)
    nbytes = logit_bytes(w)

    target_h = torch.from_numpy(w["target"]).to(torch.bfloat16).pin_memory()
    draft_h = torch.from_numpy(w["draft"]).to(torch.bfloat16).pin_memory()
    tokens_h = torch.from_numpy(w["tokens"]).pin_memory()
    target = target_h.to(dev)
    draft = draft_h.to(dev)
    tokens = tokens_h.to(dev)
    tp = torch.from_numpy(w["target_temperature"]).to(dev)
    tq = torch.from_numpy(w["draft_temperature"]).to(dev)
    stream = torch.cuda.current_stream(dev)
    filters = {k: torch.from_numpy(v).to(dev) for k, v in w.get("filters", {}).items()}

    def step():
        return sv.verify_chain(target, draft, tokens, tp, tq, seed=seed, **filters)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()

    # device-timed region: per-call events on the launching stream, and events
    # the library records around its rows kernel (the dominant kernel)
    lib = sv.api._abi.load()

    def events(n):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in ev:
            e.record(stream)  # created now, before the library records them
        return ev

    starts, ends = events(args.steps), events(args.steps)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_begin = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_begin.record(stream)
        for i in range(args.steps):
            starts[i].record(stream)
            r = step()
            ends[i].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    elapsed_ms = max_over_ranks(t_begin.elapsed_time(t_end), world, dev)
    call_ms = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
    # the dominant kernel alone: a second timed loop of the same calls in which
    # the library records events around its rows kernel (kept out of the loop
    # above: events between the kernels hold back the next kernel's early
    # launch, which the headline number should not pay for)
    k_steps = min(args.steps, 500)
    k_starts, k_ends = events(k_steps), events(k_steps)
    torch.cuda.synchronize()
    for i in range(k_steps):
        lib.spec_set_profile_events(k_starts[i].cuda_event, k_ends[i].cuda_event)
        step()
    torch.cuda.synchronize()
    lib.spec_set_profile_events(None, None)
    kernel_ms = [s_.elapsed_time(e_) for s_, e_ in zip(k_starts, k_ends)]
    ms_per_step = elapsed_ms / args.steps
    value = job_rate(world, rows, args.steps, elapsed_ms / 1e3)
    clocks = clocks_of(clk, local, step)

    # what the pages ask a verifier to report beside its speed: the accepted
    # length per target invocation and the per-position acceptance rate beta
    n_acc = r.num_accepted.to("cpu").numpy()
    acceptance = {"mean_emitted_tokens": float(np.mean(n_acc + 1)),
                  "mean_accepted_drafts": float(np.mean(n_acc))}
    if not filters:  # beta of the unfiltered distributions
        beta = sv.overlap(target, draft, tp, tq).beta.to("cpu").numpy()
        acceptance["mean_beta_per_position"] = [round(float(x), 4) for x in beta.mean(axis=0)]
        acceptance["mean_beta"] = float(beta.mean())

    # end to end through the binding: pinned host inputs in, results back out;
    # one untimed step first, in which the device buffers the copies land in
    # are allocated (every timed step still copies its inputs and reads back)
    def e2e_step():
        t_d = target_h.to(dev, non_blocking=True)
        d_d = draft_h.to(dev, non_blocking=True)
        k_d = tokens_h.to(dev, non_blocking=True)
        r2 = sv.verify_chain(t_d, d_d, k_d, tp, tq, seed=seed, **filters)
        return r2.num_accepted.to("cpu"), r2.tokens.to("cpu")

    e2e_steps = max(1, args.e2e_steps)
    e2e_step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        n_out, t_out = e2e_step()
    torch.cuda.synchronize()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / e2e_steps, world, dev)
    h2d = target_h.numel() * 2 + draft_h.numel() * 2 + tokens_h.numel() * 4
    d2h = n_out.numel() * 4 + t_out.numel() * 4
    # the same host-to-device copies alone: what the end-to-end number can reach
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        t_d = target_h.to(dev, non_blocking=True)
        d_d = draft_h.to(dev, non_blocking=True)
        k_d = tokens_h.to(dev, non_blocking=True)
    torch.cuda.synchronize()
    copy_s = (time.perf_counter() - t0) / e2e_steps

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    # a sample of the timed calls checked against the oracle (same seed)
    n_check = min(B, 8)
    from oracle import verify as ov
    want = ov.verify_chain(w["target"], w["draft"], w["tokens"], w["target_temperature"],
                           w["draft_temperature"], seed=seed, seqs=range(n_check),
                           **w.get("filters", {}))
    got_n, got_t = r.num_accepted.to("cpu").numpy(), r.tokens.to("cpu").numpy()
    mismatched = sum(1 for b, o in enumerate(want)
                     if got_n[b] != o["num_accepted"] or list(got_t[b]) != o["tokens"])

    avg_call_ms = statistics.mean(call_ms)
    avg_kernel_ms = statistics.mean(kernel_ms)
    peak, peak_kind = measured_peak()
    achieved = nbytes / (avg_kernel_ms / 1e3) / 1e9
    kernel = ("chain_rows_kernel (every logit row read once; timed by CUDA "
              "events the library records around it on the call's stream, "
              f"{k_steps} calls after the headline loop)")
    if filters:
        # the rows kernel also writes the block maxima the filter kernel reads;
        # the traffic record is for the unfiltered call
        traffic = None
        launches = FILTER_LAUNCHES_PER_STEP
    else:
        # the record is for the full-size workload only
        traffic = None if args.batch else recorded_traffic()
        launches = LAUNCHES_PER_STEP
    kmed = statistics.median(kernel_ms)
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_entry(w),
        "clocks": clocks,
        "e2e": {"value": job_rate(world, rows, 1, e2e_s), "unit": "rows/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "h2d_copy_alone_gbs": h2d / copy_s / 1e9,
                "h2d_copy_alone_ms": 1e3 * copy_s},
        "gpu_launches": launches * args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "kernel": kernel,
                     "launch_ms_avg": avg_kernel_ms,
                     "launch_ms_median": kmed},
        "whole_call": {"ms_avg": avg_call_ms, "achieved_gbs": nbytes / (avg_call_ms / 1e3) / 1e9,
                       "frac_of_peak": nbytes / (avg_call_ms / 1e3) / 1e9 / peak,
                       "frac_of_8tbs_nominal": nbytes / (avg_call_ms / 1e3) / 1e9 / 8000.0},
        "acceptance": acceptance,
        "parity_sample": {"sequences": n_check, "mismatched": mismatched,
                          "against": "the CPU oracle, same inputs and seed"},
    }
    if not args.no_cpu_baseline:
        rate, dt, passes = oracle_sample_rate(w, args.cpu_seqs, min_s=10.0, max_passes=8)
        n_all = min(B, max(args.cpu_seqs, 64))
        rate_all, dt_all, procs, passes_all = oracle_all_cores(w, n_all, min_s=8.0)
        line["cpu_baseline"] = {"value": rate_all, "unit": "rows/s", "cores": procs,
                                "kind": "oracle",
                                "sample": f"{passes_all} passes over the first {n_all} of {B} "
                                          f"sequences split over {procs} processes "
                                          f"({os.cpu_count()} host cores), {dt_all:.1f} s",
                                "one_core": {"value": rate, "cores": 1,
                                             "sample": f"{passes} passes over the first "
                                                       f"{args.cpu_seqs} of {B} sequences, "
                                                       f"{dt:.1f} s"}}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def overlap_bytes(w):
    """Algorithmic bytes of one overlap call: each (target, draft) row pair of
    the gamma draft positions read once (the bonus row is not read)."""
    esize = 2 if w["dtype"] == "bf16" else 4
    return 2 * w["B"] * w["gamma"] * w["V"] * esize


def overlap_config(w):
    c = config_entry(w)
    c["workload"] = (f"overlap beta B={w['B']} gamma={w['gamma']} V={w['V']} {w['dtype']} "
                     "(temperature 1, Zipf logits, draft sigma 0.4)")
    c["row_pair_bytes_per_step"] = overlap_bytes(w)
    c["l2"] = l2_note(overlap_bytes(w), "row pairs")
    return c


def oracle_overlap_rate(w, n_seqs):
    """The CPU oracle's beta on the first n_seqs sequences: (positions/s, seconds)."""
    from oracle import verify as ov
    t0 = time.perf_counter()
    ov.chain_overlap(w["target"][:n_seqs], w["draft"][:n_seqs], w["target_temperature"][:n_seqs],
                     w["draft_temperature"][:n_seqs])
    dt = time.perf_counter() - t0
    return n_seqs * w["gamma"] / dt, dt


def typical_bytes(w):
    """Algorithmic bytes of one typical-acceptance call: every target row once."""
    esize = 2 if w["dtype"] == "bf16" else 4
    return w["B"] * (w["gamma"] + 1) * w["V"] * esize


def typical_config(w):
    c = config_entry(w)
    c["workload"] = (f"typical acceptance B={w['B']} gamma={w['gamma']} V={w['V']} {w['dtype']} "
                     f"(epsilon {TYPICAL_EPS}, delta {TYPICAL_DELTA}, temperature 1, Zipf logits)")
    c["target_bytes_per_step"] = typical_bytes(w)
    c["l2"] = l2_note(typical_bytes(w), "target rows")
    return c


def oracle_typical_rate(w, n_seqs):
    """The CPU oracle's typical acceptance on the first n_seqs sequences: (rows/s, seconds)."""
    from oracle import verify as ov
    t0 = time.perf_counter()
    ov.typical_chain(w["target"], w["tokens"], w["target_temperature"], TYPICAL_EPS,
                     TYPICAL_DELTA, seqs=range(n_seqs))
    dt = time.perf_counter() - t0
    return n_seqs * (w["gamma"] + 1) / dt, dt


# what --op overlap / --op typical measure: metric, unit, units per call,
# algorithmic bytes, configuration, traffic record and kernel source, kernel
# launches per call, the oracle's rate and a label for the roofline kernel
ROW_OPS = {
    "overlap": dict(metric=OVERLAP_METRIC, unit="positions/s",
                    units=lambda w: w["B"] * w["gamma"], nbytes=overlap_bytes,
                    config=overlap_config, traffic=(OVERLAP_TRAFFIC_FILE, "overlap.cu"),
                    launches=1, oracle=oracle_overlap_rate,
                    kernel="overlap_kernel (timed per call)"),
    "typical": dict(metric=TYPICAL_METRIC, unit="rows/s",
                    units=lambda w: w["B"] * (w["gamma"] + 1), nbytes=typical_bytes,
                    config=typical_config, traffic=(TYPICAL_TRAFFIC_FILE, "chain_rows.cu"),
                    launches=3, oracle=oracle_typical_rate,
                    kernel="chain_rows_kernel (typical records) + typical_merge_kernel + "
                           "typical_decide_kernel (timed per call)"),
}


def run_rowop_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    op = ROW_OPS[args.op]
    w = bench_workload(args)
    # one sequence per step: a bounded sample of the same workload
    op["oracle"](w, 1)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        op["oracle"](w, 1)
    dt = time.perf_counter() - t0
    per_seq = op["units"](w) // w["B"]
    value = per_seq * args.steps / dt
    line = {
        "impl": "reference", "metric": op["metric"], "value": value, "unit": op["unit"],
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": op["config"](w),
        "cpu_baseline": {"value": value, "unit": op["unit"], "cores": 1, "kind": "oracle",
                         "sample": f"the first sequence of {w['B']} per step"},
        "e2e": {"value": value, "unit": op["unit"], "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_rowop(args):
    import torch
    import torch.distributed as dist

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_verification_temp_gb300 as sv

    op = ROW_OPS[args.op]
    w = bench_workload(args)
    B = w["B"]
    units = op["units"](w)
    nbytes = op["nbytes"](w)
    target_h = torch.from_numpy(w["target"]).to(torch.bfloat16).pin_memory()
    draft_h = torch.from_numpy(w["draft"]).to(torch.bfloat16).pin_memory()
    tokens_h = torch.from_numpy(w["tokens"]).pin_memory()
    target, draft, tokens = target_h.to(dev), draft_h.to(dev), tokens_h.to(dev)
    tp = torch.from_numpy(w["target_temperature"]).to(dev)
    tq = torch.from_numpy(w["draft_temperature"]).to(dev)
    stream = torch.cuda.current_stream(dev)

    def call(t, d, k):
        if args.op == "overlap":
            r = sv.overlap(t, d, tp, tq)
            return r.beta
        r = sv.typical_accept(t, k, tp, TYPICAL_EPS, TYPICAL_DELTA)
        return r.tokens

    for _ in range(max(args.warmup, 3)):
        call(target, draft, tokens)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_begin = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_begin.record(stream)
        for i in range(args.steps):
            starts[i].record(stream)
            call(target, draft, tokens)
            ends[i].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    elapsed_ms = max_over_ranks(t_begin.elapsed_time(t_end), world, dev)
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    clocks = clocks_of(clk, local, lambda: call(target, draft, tokens))

    # end to end: the inputs the op reads copied from pinned host memory, the
    # result read back (after one untimed step that allocates the device
    # buffers the copies land in)
    def e2e_step():
        t_d = target_h.to(dev, non_blocking=True)
        if args.op == "overlap":
            return call(t_d, draft_h.to(dev, non_blocking=True), None).to("cpu")
        return call(t_d, None, tokens_h.to(dev, non_blocking=True)).to("cpu")

    e2e_steps = max(1, args.e2e_steps)
    out = e2e_step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        out = e2e_step()
    torch.cuda.synchronize()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / e2e_steps, world, dev)
    h2d = target_h.numel() * 2 + (draft_h.numel() * 2 if args.op == "overlap"
                                  else tokens_h.numel() * 4)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    avg_launch_ms = statistics.mean(launch_ms)
    peak, peak_kind = measured_peak()
    achieved = nbytes / (avg_launch_ms / 1e3) / 1e9
    line = {
        "metric": op["metric"], "value": job_rate(world, units, args.steps, elapsed_ms / 1e3),
        "unit": op["unit"], "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": op["config"](w),
        "clocks": clocks,
        "e2e": {"value": job_rate(world, units, 1, e2e_s), "unit": op["unit"],
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": out.numel() * 4},
        "gpu_launches": op["launches"] * args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": None if args.batch else recorded_traffic(*op["traffic"]),
                     "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "kernel": op["kernel"], "launch_ms_avg": avg_launch_ms,
                     "launch_ms_median": statistics.median(launch_ms)},
    }
    if not args.no_cpu_baseline:
        n = min(B, args.cpu_seqs)
        rate, dt = op["oracle"](w, n)
        line["cpu_baseline"] = {"value": rate, "unit": op["unit"], "cores": 1, "kind": "oracle",
                                "sample": f"the first {n} of {B} sequences, {dt:.1f} s"}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


RERANK_METRIC = "reranked draft trees/s"
RERANK_T, RERANK_N, RERANK_M = 256, 1024, 64


def rerank_workload():
    from speculative_decoding_verification_temp_gb300 import workloads
    return workloads.make_rerank(RERANK_T, RERANK_N, seed=1100)


def rerank_config():
    return {"workload": f"EAGLE-2 rerank: {RERANK_T} trees of {RERANK_N} nodes, top m = {RERANK_M}",
            "T": RERANK_T, "N": RERANK_N, "m": RERANK_M,
            "input_bytes_per_step": RERANK_T * RERANK_N * 8,
            "l2": "L2 flushed (a 256 MB write) before every call; value from the calls' own "
                  "event times"}


def oracle_rerank_rate(w, n_trees):
    from oracle import verify as ov
    t0 = time.perf_counter()
    for t in range(n_trees):
        ov.tree_rerank(w["parent"][t], w["confidence"][t], RERANK_M)
    dt = time.perf_counter() - t0
    return n_trees / dt, dt


def run_rerank(args):
    world, rank, local = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return
        w = rerank_workload()
        oracle_rerank_rate(w, 1)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            oracle_rerank_rate(w, 1)
        dt = time.perf_counter() - t0
        value = args.steps / dt
        print(json.dumps({
            "impl": "reference", "metric": RERANK_METRIC, "value": value, "unit": "trees/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": rerank_config(),
            "cpu_baseline": {"value": value, "unit": "trees/s", "cores": 1, "kind": "oracle",
                             "sample": "one tree per step"},
            "e2e": {"value": value, "unit": "trees/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}), flush=True)
        return
    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_verification_temp_gb300 as sv

    w = rerank_workload()
    par_h = torch.from_numpy(w["parent"]).pin_memory()
    conf_h = torch.from_numpy(w["confidence"]).pin_memory()
    par, conf = par_h.to(dev), conf_h.to(dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(args.warmup, 3)):
        sv.tree_rerank(par, conf, RERANK_M)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_begin = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_begin.record(stream)
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            sv.tree_rerank(par, conf, RERANK_M)
            ends[i].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    elapsed_ms = max_over_ranks(sum(launch_ms), world, dev)
    clocks = clocks_of(clk, local, lambda: sv.tree_rerank(par, conf, RERANK_M))
    # end to end (after one untimed step that allocates the device buffers)
    def e2e_step():
        r = sv.tree_rerank(par_h.to(dev, non_blocking=True), conf_h.to(dev, non_blocking=True),
                           RERANK_M)
        return r.nodes.to("cpu")

    e2e_steps = max(1, args.e2e_steps)
    out = e2e_step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        out = e2e_step()
    torch.cuda.synchronize()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / e2e_steps, world, dev)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    avg_launch_ms = statistics.mean(launch_ms)
    peak, peak_kind = measured_peak()
    nbytes = RERANK_T * RERANK_N * 8 + RERANK_T * RERANK_M * 12 + RERANK_T * 8
    achieved = nbytes / (avg_launch_ms / 1e3) / 1e9
    line = {
        "metric": RERANK_METRIC, "value": job_rate(world, RERANK_T, args.steps, elapsed_ms / 1e3),
        "unit": "trees/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": rerank_config(),
        "clocks": clocks,
        "e2e": {"value": job_rate(world, RERANK_T, 1, e2e_s), "unit": "trees/s",
                "h2d_bytes_per_step": (par_h.numel() + conf_h.numel()) * 4,
                "d2h_bytes_per_step": out.numel() * 4},
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "kernel": "tree_rerank_kernel (latency-bound: one CTA per tree, "
                               "log-depth and per-level passes, a bitonic sort)",
                     "launch_ms_avg": avg_launch_ms,
                     "launch_ms_median": statistics.median(launch_ms)},
    }
    if not args.no_cpu_baseline:
        n = min(RERANK_T, args.cpu_seqs)
        rate, dt = oracle_rerank_rate(w, n)
        line["cpu_baseline"] = {"value": rate, "unit": "trees/s", "cores": 1, "kind": "oracle",
                                "sample": f"{n} of {RERANK_T} trees, {dt:.1f} s"}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_workloads(args):
    """Per-call device times of the five verification workloads (plus workload
    2 with top-p 0.9 and min-p 0.05) and the tree mask: CUDA events around each
    call through the Python API, every input (logits, tokens, temperatures,
    filter arrays) resident on the device before the timing, the L2 flushed (a
    256 MB write) and the GPU held busy for about 100 us before every call so
    that the binding's host work is done before the first kernel starts; the
    median of --steps calls after --warmup calls.  One JSON line with every
    workload."""
    import torch
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_verification_temp_gb300 as sv
    from speculative_decoding_verification_temp_gb300 import workloads

    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def median_call_us(fn):
        for _ in range(max(args.warmup, 3)):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(args.steps):
            flush.zero_()
            torch.cuda._sleep(200_000)  # the host queues the call meanwhile
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1e3)
        return statistics.median(ts)

    def dev_logits(x, dtype):
        t = torch.from_numpy(x).to(dev)
        return t.to(torch.bfloat16) if dtype == "bf16" else t

    def top_k(x):
        # only a real filter is passed (any top-k array routes the call to the
        # kernels that apply top-k), as a device array
        return torch.from_numpy(x).to(dev) if x is not None and (x > 0).any() else None

    def on_dev(x):
        return torch.from_numpy(np.ascontiguousarray(x)).to(dev)

    per = {}
    ids = [int(x) for x in args.only.split(",")] if args.only else range(5)
    for i in ids:
        w = workloads.config(i)
        t = dev_logits(w["target"], w["dtype"])
        d = dev_logits(w["draft"], w["dtype"])
        esize = 2 if w["dtype"] == "bf16" else 4
        tp, tq = on_dev(w["target_temperature"]), on_dev(w["draft_temperature"])
        kp, kq = top_k(w.get("target_top_k")), top_k(w.get("draft_top_k"))
        tok = torch.from_numpy(w["tokens"]).to(dev)
        if "B" in w:
            us = median_call_us(lambda: sv.verify_chain(t, d, tok, tp, tq, kp, kq, seed=w["seed"]))
            rows = w["B"] * (w["gamma"] + 1)
            if i == 2:
                fp = torch.full((w["B"],), FILTER_TOP_P, dtype=torch.float32, device=dev)
                fm = torch.full((w["B"],), FILTER_MIN_P, dtype=torch.float32, device=dev)
                fus = median_call_us(lambda: sv.verify_chain(
                    t, d, tok, tp, tq, seed=w["seed"], target_top_p=fp, draft_top_p=fp,
                    target_min_p=fm, draft_min_p=fm))
                per["workload_2_filters"] = {
                    "us_per_call": fus, "rows_per_s": rows / (fus / 1e6), "dtype": w["dtype"],
                    "V": w["V"], "esize": esize,
                    "filters": f"top-p {FILTER_TOP_P} and min-p {FILTER_MIN_P}, both sides"}
        else:
            par = torch.from_numpy(w["parent"]).to(dev)
            us = median_call_us(lambda: sv.verify_tree(
                t, d, tok, par, w["max_depth"], tp, tq, kp, kq, seed=w["seed"]))
            rows = w["T"] * w["N"]
            per["tree_mask"] = {"us_per_call": median_call_us(
                lambda: sv.tree_mask(par, w["max_depth"])), "trees": w["T"], "nodes": w["N"]}
        per[f"workload_{i}"] = {"us_per_call": us, "rows_per_s": rows / (us / 1e6),
                                "dtype": w["dtype"], "V": w["V"], "esize": esize}
    print(json.dumps({"metric": "per-call time of each workload", "unit": "us",
                      "steps": args.steps, "warmup": args.warmup, "data": "synthetic",
                      "l2": "flushed (a 256 MB write) before every call",
                      "timing": "device time: inputs on the device, the GPU busy while the "
                                "host queues each call",
                      "workloads": per}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-seqs", type=int, default=256)
    ap.add_argument("--reference-seqs", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=0,
                    help="sequences per batch (default: the B = 256 workload); for profiling")
    ap.add_argument("--op", default="verify",
                    choices=["verify", "filters", "overlap", "typical", "rerank", "workloads"],
                    help="verify: the chain verifier (default); filters: the same with top-p "
                         "0.9 and min-p 0.05; overlap: beta_i per position; "
                         "typical: typical acceptance; rerank: EAGLE-2 tree rerank; "
                         "workloads: per-call times of workloads 0-4 and the tree mask")
    ap.add_argument("--only", default="",
                    help="--op workloads: a comma list of workload ids (default: 0-4)")
    args = ap.parse_args()
    if args.op == "workloads":
        run_workloads(args)
    elif args.op == "rerank":
        run_rerank(args)
    elif args.op in ROW_OPS:
        if args.impl == "reference":
            run_rowop_reference(args)
        else:
            run_rowop(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
