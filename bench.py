#!/usr/bin/env python3
"""Throughput of the batched verify-and-sample epilogue on one or more GB300s.

One step = one call of the whole epilogue (penalties, temperature, top-k / top-p on target
and draft, acceptance, residual / bonus draws, logprobs) over one batch of the
B=64, K=8, V=262,144 workload (bf16 logits, fp32 draft probabilities, inputs resident in
HBM; 839 MB per batch, larger than the 129 MB L2, so no flush is needed between steps).

Prints one JSON line: verify rows/s (whole job) of the call as shipped, the streaming
kernel's roofline (timed in a second loop with events around it), clocks seen during the
timed region, an end-to-end figure through the host-buffer entry point, the float64 oracle
timed on all host cores over the whole batch (and on one thread over a sample), and the
parity of the timed call's results with the oracle's, near ties counted.  On one GPU it also
times, with their parity, the same call on the workload's draft-layout variants (one-hot
lookup drafts; a reduced draft vocabulary) and with every option of dspark_extras_t on.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "b64k8v262144"
METRIC = "verify rows/s & HBM GB/s (% roofline), B=64 K=8 V=262144 bf16, 1×GB300"
UNIT = "verify rows/s"
DOMINANT = "stream_stats_kernel"
CPU_SAMPLE_S = 10.0                   # seconds of one-thread oracle work in the native arm's cpu_baseline
NOMINAL_HBM_GBS = 8000.0              # the ~8 TB/s HBM3e figure the roofline target is stated against
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "stream_stats_kernel_b64k8v262144.md")
KERNEL_SOURCES = [os.path.join(ROOT, "sample_verify_epilogue_gb300", "csrc", f)
                  for f in ("stream_stats.cu", "dspark_internal.cuh")]


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic():
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary, or None
    when the summary is missing or was taken on a different kernel source."""
    try:
        txt = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    vals = {}
    for ln in txt.splitlines():
        ln = ln.strip().lstrip("-* ")
        if ":" in ln and ln.startswith(("traffic_bytes_per_launch", "kernel_source_hash")):
            k, v = ln.split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_hash") != kernel_source_hash():
        return None
    try:
        return float(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self, t0, t1):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        for ln in open(self.path):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        inside = [r for r in rows if t0 - 1.0 <= r[0] <= t1 + 1.0] or rows
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


class DriverEvents:
    """CUDA events created and read through the driver API.  The library records them on the
    launching stream right around the streaming kernel (torch's Event refuses events that
    torch itself did not record)."""

    def __init__(self, n):
        import ctypes
        self.ct = ctypes
        self.cu = ctypes.CDLL("libcuda.so.1")
        self.cu.cuEventCreate.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_uint]
        self.cu.cuEventElapsedTime_v2.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_void_p, ctypes.c_void_p]
        self.cu.cuEventDestroy_v2.argtypes = [ctypes.c_void_p]
        self.pairs = []
        for _ in range(n):
            a, b = ctypes.c_void_p(), ctypes.c_void_p()
            assert self.cu.cuEventCreate(ctypes.byref(a), 0) == 0
            assert self.cu.cuEventCreate(ctypes.byref(b), 0) == 0
            self.pairs.append((a.value, b.value))

    def ms(self, i):
        out = self.ct.c_float()
        rc = self.cu.cuEventElapsedTime_v2(self.ct.byref(out), self.pairs[i][0], self.pairs[i][1])
        assert rc == 0, rc
        return float(out.value)

    def close(self):
        for a, b in self.pairs:
            self.cu.cuEventDestroy_v2(a)
            self.cu.cuEventDestroy_v2(b)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def workload_config(ws):
    """The `config` object of both arms' JSON lines: the bench workload and its settings."""
    return {"workload": WORKLOAD, "B": 64, "K": 8, "V": 262144,
            "logits": "bf16", "q": "fp32", "T": 1.0, "top_k": 64, "top_p": 0.95,
            "penalties": "presence 0.2 / frequency 0.2, 4096-token Zipf histories",
            "top_logprobs": 20, "l2": "inputs (839 MB) larger than L2, no flush",
            "parallelism": f"{ws} independent replica(s), no collective"}


def whole_job_rate(dist, local_ms, units_per_rank_step, steps, ws, device=None):
    """Whole-job throughput: the units every rank processed over the slowest rank's time
    (max over ranks).  Returns (rate per second, that time in ms)."""
    if dist is not None:
        import torch
        t = torch.tensor([float(local_ms)], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        local_ms = float(t.item())
    return units_per_rank_step * steps * ws / (local_ms / 1e3), local_ms


def time_oracle(batch, requests):
    from oracle import epilogue as O
    t = time.perf_counter()
    O.verify_batch(batch, requests)
    return time.perf_counter() - t


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _pool_ready(_):
    import numpy  # noqa: F401  (worker start-up: imports done before the timed map)
    from oracle import epilogue  # noqa: F401
    return os.getpid()


def _oracle_outcomes(sub):
    """Worker: the oracle's outcomes of every request of a (small) batch."""
    from oracle import epilogue as O
    return [O.outcomes(sub, i) for i in range(sub.B)]


class OraclePool:
    """The float64 oracle on all host cores: a spawn-started process pool (never forked
    from a process that has touched the GPU), one request per task."""

    def __init__(self, n=None):
        import multiprocessing as mp
        from concurrent.futures import ProcessPoolExecutor
        self.n = n or host_cores()
        self.ex = ProcessPoolExecutor(max_workers=self.n, mp_context=mp.get_context("spawn"))
        list(self.ex.map(_pool_ready, range(4 * self.n)))

    def outcomes(self, batch, requests):
        """({b: outcomes}, wall seconds) for the given requests of batch."""
        subs = [batch.subset([b]) for b in requests]
        t = time.perf_counter()
        res = list(self.ex.map(_oracle_outcomes, subs, chunksize=1))
        el = time.perf_counter() - t
        return {b: r[0] for b, r in zip(requests, res)}, el

    def close(self):
        self.ex.shutdown()


VARIANTS = (
    ("b64k8v262144_onehot", None),
    ("b64k8v262144_d2t32000", None),
    ("b64k8v262144", "options"),
)


def measure_variant(name, option, steps, device, pool):
    """ms per call, verify rows/s, algorithmic GB/s of the call and of the streaming kernel
    (events around it, as in the headline), and parity with the oracle on every request, for
    one variant of the workload."""
    import dataclasses

    import numpy as np
    import torch

    from sample_verify_epilogue_gb300.runner import EpilogueCall
    from tests._compare import compare
    from workloads import configs

    batch = configs.build(name)
    label = name
    if option == "options":
        # eos = each request's draft 3, per-position counters, penalised logprobs
        batch = dataclasses.replace(batch, eos_ids=batch.draft_ids[:, 3].copy(), logprob_mode="penalised")
        label = name + " +eos +counters +penalised logprobs"
    call = EpilogueCall(batch, device=device, counters=True)
    stream = torch.cuda.current_stream(device)
    for _ in range(5):
        call.run()
    torch.cuda.synchronize(device)
    call.pos_counts.zero_()
    call.run()
    res = call.results()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        call.run()
    t1.record(stream)
    torch.cuda.synchronize(device)
    ms = t0.elapsed_time(t1) / steps
    kn = max(1, min(steps, 100))
    ev = DriverEvents(kn)
    for i in range(kn):
        call.run(stage_events=ev.pairs[i])
    torch.cuda.synchronize(device)
    kern_ms = statistics.mean(ev.ms(i) for i in range(kn))
    ev.close()
    outs, _ = pool.outcomes(batch, range(batch.B))
    tally = compare(batch, res, outs)
    counters_ok = bool(np.array_equal(res["pos_counts"][0], tally.attempted) and
                       np.array_equal(res["pos_counts"][1], tally.accepted))
    algo = batch.algorithmic_bytes()
    del call
    torch.cuda.empty_cache()
    return {"workload": label, "q_layout": batch.q_layout, "draft_row_len": batch.draft_row_len(),
            "ms_per_step": ms, "value": batch.verify_rows() / (ms / 1e3), "unit": UNIT,
            "algorithmic_bytes_per_step": algo, "call_gbs": algo / (ms / 1e3) / 1e9,
            "kernel_ms": kern_ms, "kernel_gbs": algo / (kern_ms / 1e3) / 1e9,
            "parity": {"requests": tally.requests, "matched": tally.requests, "single_result": tally.single,
                       "near_tie_decisions": dict(tally.near_ties), "stopped": tally.stopped,
                       "counters_match": counters_ok}}


def run_reference(args):
    ws, rank, _ = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        if rank != 0:
            dist.destroy_process_group()
            return
    from workloads import configs
    pool = OraclePool()
    # each step: as many requests of the workload as there are host cores, one per core
    nb = configs.build_size(WORKLOAD)
    wanted = [[(i * pool.n + k) % nb for k in range(pool.n)] for i in range(args.warmup + args.steps)]
    needed = sorted({b for reqs in wanted for b in reqs})
    batch = configs.build(WORKLOAD, requests=needed)        # only the requests the steps use
    steps = [[needed.index(b) for b in reqs] for reqs in wanted]
    for reqs in steps[:args.warmup]:
        pool.outcomes(batch, reqs)
    el, rows = 0.0, 0
    for reqs in steps[args.warmup:]:
        _, t = pool.outcomes(batch, reqs)
        el += t
        rows += int(sum(int(batch.rows["num_drafts"][b]) + 1 for b in reqs))
    pool.close()
    value = rows / el
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": pool.n, "kind": "oracle",
                         "sample": f"{pool.n} requests ({rows // args.steps} verify rows) of the workload per step, "
                                   f"one per host core, float64 numpy oracle in a spawn-started process pool"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_native(args):
    import numpy as np
    import torch

    import __graft_entry__
    from sample_verify_epilogue_gb300 import binding
    from sample_verify_epilogue_gb300.runner import EpilogueCall
    from workloads import configs

    ws, rank, local = dist_env()
    dist = None
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if rank == 0 or ws == 1:
        __graft_entry__.build()
    if dist is not None:
        dist.barrier()
    binding.load_library()

    # each rank owns its own 64 requests (independent problems: weak scaling, no collective)
    batch = configs.build(WORKLOAD)
    call = EpilogueCall(batch, device=device)
    stream = torch.cuda.current_stream(device)
    kern_steps = max(1, min(args.steps, 200))
    stage_ev = DriverEvents(kern_steps)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)

    for _ in range(args.warmup):
        call.run()
    torch.cuda.synchronize(device)
    res = call.results()
    accepted = int(np.sum(res["accept_len"].astype(np.int64) + 1))

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(device)
    w0 = time.time()
    # the timed region: the shipped call, back to back, nothing else on the stream
    t_start.record(stream)
    for i in range(args.steps):
        call.run()
    t_end.record(stream)
    torch.cuda.synchronize(device)
    if dist is not None:
        dist.barrier()
    elapsed_ms = t_start.elapsed_time(t_end)
    # the streaming kernel on its own: a second loop with events recorded right around it
    # (the events cost the call its programmatic launch overlap around that kernel)
    for i in range(kern_steps):
        call.run(stage_events=stage_ev.pairs[i])
    torch.cuda.synchronize(device)
    w1 = time.time()
    clocks = sampler.stop(w0, w1) if sampler else None
    kern_ms = statistics.mean(stage_ev.ms(i) for i in range(kern_steps))
    stage_ev.close()
    rows_per_step = batch.verify_rows()
    algo_bytes = batch.algorithmic_bytes()
    value, elapsed_ms = whole_job_rate(dist, elapsed_ms, rows_per_step, args.steps, ws, device)
    peak, peak_kind = peaks()
    achieved = algo_bytes / (kern_ms / 1e3) / 1e9
    traffic = measured_traffic()

    # end to end through the host-buffer entry point: pinned inputs in, results out, every step
    e2e = None
    if rank == 0 or ws > 1:
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
        hx = pin(np.ascontiguousarray(batch.x).view(np.int16))
        hq = pin(batch.q)
        hd = pin(batch.draft_ids)
        hrows = pin(np.ascontiguousarray(batch.rows).view(np.uint8))
        hcounts = (pin(batch.hist_offsets), pin(batch.hist_ids), pin(batch.hist_counts))
        hu = pin(batch.uniforms)
        W = batch.K_max + 1
        hout = {"accept_len": torch.empty(batch.B, dtype=torch.int32).pin_memory(),
                "tokens": torch.empty(batch.B, W, dtype=torch.int32).pin_memory(),
                "logprobs": torch.empty(batch.B, W, dtype=torch.float32).pin_memory(),
                "top_ids": torch.empty(batch.B, W, batch.n_top_logprobs, dtype=torch.int32).pin_memory(),
                "top_logprobs": torch.empty(batch.B, W, batch.n_top_logprobs, dtype=torch.float32).pin_memory()}
        hst = torch.empty(batch.B, dtype=torch.int32).pin_memory()
        nbytes = binding.dspark_host_workspace_bytes(batch.B, batch.K_max, batch.V, "bf16", batch.n_top_logprobs,
                                                     int(batch.hist_offsets[-1]))
        del call
        torch.cuda.empty_cache()
        hws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        sid = stream.cuda_stream

        def host_call():
            binding.dspark_verify_sample_host(hx, hq, hd, hcounts, hrows, hu, out=hout, row_status=hst,
                                              workspace=hws, logits_dtype="bf16", want_logprobs=True,
                                              n_top_logprobs=batch.n_top_logprobs, stream=sid)

        e2e_steps = max(1, min(args.steps, 200))
        for _ in range(max(1, min(args.warmup, 5))):
            host_call()
        t = time.perf_counter()
        for _ in range(e2e_steps):
            host_call()
        el = time.perf_counter() - t
        h2d = sum(int(a.numel() * a.element_size()) for a in (hx, hq, hd, hrows, hu, *hcounts))
        d2h = sum(int(a.numel() * a.element_size()) for a in (*hout.values(), hst))
        e2e = {"value": rows_per_step * e2e_steps * ws / el, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
        assert np.array_equal(hout["accept_len"].numpy(), res["accept_len"])

    cpu = parity = None
    variants = None
    if rank == 0 and ws == 1:
        # the oracle on every request of this very batch, all host cores (spawn-started pool):
        # the all-cores baseline, and the parity of the timed call's results with the oracle
        from tests._compare import compare
        pool = OraclePool()
        outs, wall = pool.outcomes(batch, range(batch.B))
        peak_v, _ = peaks()
        variants = []
        for name, option in VARIANTS:
            v = measure_variant(name, option, max(1, min(args.steps, 500)), device, pool)
            v["kernel_frac"] = v["kernel_gbs"] / peak_v
            variants.append(v)
        pool.close()
        tally = compare(batch, res, outs)
        parity = {"requests": tally.requests, "matched": tally.requests, "single_result": tally.single,
                  "decisions": tally.decisions, "near_tie_decisions": dict(tally.near_ties),
                  "near_tie_requests": tally.near_tie_requests, "off_float64": tally.off_float64,
                  "eps": 1e-6, "logprob_tol": 1e-4}
        # one host thread, on requests of the same batch one after another, for about 10 s
        n_req, t = 0, 0.0
        while n_req < batch.B and (n_req == 0 or t < CPU_SAMPLE_S):
            t += time_oracle(batch, [n_req])
            n_req += 1
        rows_done = int(sum(int(batch.rows[b]["num_drafts"]) + 1 for b in range(n_req)))
        cpu = {"value": rows_per_step / wall, "unit": UNIT, "cores": pool.n, "kind": "oracle",
               "sample": f"all {batch.B} requests ({rows_per_step} verify rows) of the timed batch, float64 numpy "
                         f"oracle, one request per task on {pool.n} host cores (spawn-started process pool), "
                         f"{wall:.1f} s",
               "single_thread": {"value": rows_done / t, "unit": UNIT, "cores": 1,
                                 "sample": f"{n_req} requests ({rows_done} verify rows), one thread, {t:.1f} s"}}

    if rank == 0:
        out = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": workload_config(ws),
            "sampled_tokens_per_s": accepted * args.steps * ws / (elapsed_ms / 1e3),
            "hbm_gbs_per_call": algo_bytes * args.steps * ws / (elapsed_ms / 1e3) / 1e9 / ws,
            "algorithmic_bytes_per_step": algo_bytes,
            "roofline": {"bound": "hbm", "kernel": DOMINANT, "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_kind, "traffic": traffic,
                         "kernel_ms": kern_ms, "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                         "call_achieved": algo_bytes / (elapsed_ms / args.steps / 1e3) / 1e9,
                         "call_frac": algo_bytes / (elapsed_ms / args.steps / 1e3) / 1e9 / peak},
            "near_ties": None if parity is None else sum(parity["near_tie_decisions"].values()),
            "parity": parity,
            "gpu_launches": binding.dspark_launches_per_call() * args.steps,
            "clocks": clocks,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "variants": variants,
        }
        print(json.dumps(out))
    if dist is not None:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=("native", "reference"), default="native")
    args = ap.parse_args()
    if args.impl == "reference":
        args.steps = 10 if args.steps is None else args.steps
        args.warmup = 3 if args.warmup is None else args.warmup
        run_reference(args)
    else:
        args.steps = 2000 if args.steps is None else args.steps
        args.warmup = 20 if args.warmup is None else args.warmup
        run_native(args)


if __name__ == "__main__":
    main()
