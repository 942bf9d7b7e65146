"""SGMV LoRA benchmark: LoRA-routed tokens/s and HBM GB/s vs roofline.

One step = the SGMV delta of one batch on both problems of a layer: the
fused q/k/v projection and o_proj (gate+up and down for the MLP workload),
each one lora_sgmv_apply (shrink + boundary-aware expand).  The batch's
routing triple is built on the host (lora_build_routing) and uploaded once
when the inputs are prepared; the timed `value` region holds only the
applies.  The routing build is timed in `e2e`.

Workloads (seeded synthetic data; see workloads/synthetic.py):
  mixed70b   the N=1 line (the largest configuration): Llama-3-70B-shaped
             attention (hidden 8192, 64/8 heads, hd 128; fused qkv 10240,
             o 8192 -> 8192), 16 slots, max rank 128 (ranks 16/64/128),
             8192 tokens = 6 prefill requests of 512-1024 plus 1-token
             decodes, 20% base, bf16.
  decode8b   secondary block: Llama-3-8B decode (hidden 4096; qkv 6144,
             o 4096), 8 slots, max rank 16, 256 one-token requests, 25% base.
  prefill8b  secondary block: ragged prefill, 8B shapes, 4 slots + base,
             max rank 64, 16 requests of 128-2048 tokens.
  (many64, mlp8b: --workload only.)

value:   K steps timed exactly, with CUDA events on the launching stream,
         replayed from CUDA graphs of several steps each (floor(K/NS)
         replays of one graph over all NS input sets plus one graph of the
         remaining steps), inputs resident in HBM; NS input sets (the layers
         of one batch: own x, y, A/B each, one shared routing triple) whose
         footprint exceeds 4x L2, so each step streams from HBM.
roofline: per workload, the fused-qkv apply (the larger unit of a step)
         timed over the rotated sets in 5 trials of >= 30 ms each; achieved
         = its algorithmic bytes / its median duration.
e2e:     the main workload's steps through the Python API with host
         buffers: per step the host routing build, one pinned host->device
         copy of x, y and the triple, the two applies, one device->host copy
         of both y outputs.
cpu_baseline / --impl reference: the CPU oracle (plain C in double) on a
         bounded sample of the same workload: the OpenMP build on every core
         of the process's affinity mask, and the single-threaded build.

Run: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
     [--workload mixed70b|decode8b|prefill8b|many64|mlp8b] [--no-secondary]
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LoRA-routed tokens/sec for SGMV shrink+expand; achieved HBM GB/s vs roofline"
MAIN_WORKLOAD = "mixed70b"
SECONDARY = ("decode8b", "prefill8b")

WORKLOAD_DESC = {
    "decode8b": "decode, Llama-3-8B attention (hidden 4096, 32/8 heads, hd 128; fused qkv 6144 + o 4096), "
                "8 slots, max rank 16, 256 x 1-token requests, 25% base, bf16",
    "many64": "many-adapter decode, 8B shapes, 64 slots, rank 16, 1024 x 1-token requests, Zipf(1.1), 10% base, "
              "per-projection q/k/v + o, bf16",
    "prefill8b": "ragged prefill, 8B shapes, 4 slots + base, max rank 64, 16 requests of 128-2048 tokens, bf16",
    "mixed70b": "mixed prefill+decode, Llama-3-70B attention (hidden 8192, 64/8 heads; fused qkv 10240 + o 8192), "
                "16 slots, max rank 128, 8192 tokens, 20% base, bf16",
    "mixed64": "mixed prefill+decode over many adapters, 8B attention shapes, 64 slots, max rank 64, 3328 tokens "
               "= 4 prefill requests of 512-768 + 1-token decodes, 10% base, bf16",
    "mlp8b": "decode, Llama-3-8B MLP (hidden 4096, intermediate 14336; fused gate+up 28672 + down 4096), "
             "8 slots, max rank 16, 256 x 1-token requests, 25% base, bf16",
}


def _env_rank():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def reduce_across_ranks(max_values, sum_values, dist=None, device="cpu"):
    """Whole-job figures across replicas: the slowest rank's times (max) and
    the routed tokens of all ranks (sum).  Single process: unchanged."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return list(max_values), list(sum_values)
    import torch
    mx = torch.tensor([float(v) for v in max_values], dtype=torch.float64, device=device)
    sm = torch.tensor([float(v) for v in sum_values], dtype=torch.float64, device=device)
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    dist.all_reduce(sm, op=dist.ReduceOp.SUM)
    return mx.tolist(), sm.tolist()


def rank_seed(rank: int, index: int) -> int:
    """Seed of input set `index` on replica `rank` (replicas draw disjoint batches)."""
    return 1000 * rank + index


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _tensor_peak():
    """Dense bf16 tensor peak in TFLOP/s (burst: the apply is timed on its own)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def _names(proj):
    from workloads.synthetic import PROBLEMS
    return list(PROBLEMS[proj])


def algorithmic_bytes(route_host, raw, proj, e=2, slot_ranks=False):
    """Per-apply algorithmic bytes: routed x rows + touched A/B slots + y read+write.
    A/B count the padded rank R, or ceil16(rank) per slot when the kernels are
    given the true ranks (they then skip the rest)."""
    E = route_host["end"]
    touched = sorted(set(int(s) for s in route_host["lora_ids"]))
    names = _names(proj)
    n = len(names)
    O = sum(raw["out_dims"][nm] for nm in names)
    R = raw["max_lora_rank"]
    k = raw["in_dims"][names[0]]
    ranks = [min(R, (int(raw["rank"][s]) + 15) // 16 * 16) if slot_ranks else R for s in touched]
    return E * k * e + sum(n * r * k * e + O * r * e for r in ranks) + 2 * E * O * e


def algorithmic_flops(route_host, raw, proj):
    E = route_host["end"]
    names = _names(proj)
    O = sum(raw["out_dims"][nm] for nm in names)
    R = raw["max_lora_rank"]
    k = raw["in_dims"][names[0]]
    return E * (2 * len(names) * R * k + 2 * R * O)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


class ClockSampler:
    """nvidia-smi clocks + throttle reasons sampled every 200 ms while running;
    summarised over the samples that fall inside the marked timed regions."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []  # (arrival time, csv line)
        self.t = None
        self.windows = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        """A timed region ran from t0 to t1 (time.time())."""
        self.windows.append((t0, t1 + 0.25))

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        inside = [(t, ln) for t, ln in self.lines if any(a <= t <= b for a, b in self.windows)]
        lines = inside or self.lines
        for _, ln in lines:
            p = [v.strip() for v in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax.append(float(p[2]))
            except ValueError:
                continue
            for nm, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm),
                "window": "timed regions (the K steps and the roofline trials)" if inside else "whole run"}


# ----------------------------------------------------------------- oracle --

def oracle_step_sampler(workload, seed):
    """Prepared oracle problems and run(nrows, parallel) running the oracle on
    the first nrows routed rows of both problems.  Returns (run, end)."""
    import oracle
    from workloads import synthetic as sy

    raw = sy.draw(workload, seed)
    spec = sy.SPECS[workload]
    p0, p1 = spec.problems
    probs = [oracle.prepare_problem(raw, p0, fused=spec.fused_qkv), oracle.prepare_problem(raw, p1, fused=True)]
    end = probs[0]["end"]
    cache = {}  # converted rows (conversion is not timed)

    def run(nrows, parallel=False):
        rows = np.arange(min(nrows, end), dtype=np.int32)
        for p in probs:
            key = (id(p), rows.size)
            if key not in cache:
                x_rows = oracle.to_f64(p["x"][rows], p["dtype"])
                sl = []
                for s in p["slices"]:
                    d = dict(s)
                    d["y_in"] = oracle.to_f64(s["y"][rows][:, s["y_col0"]:s["y_col0"] + s["out_dim"]], p["dtype"])
                    sl.append(d)
                cache[key] = (x_rows, sl)
            x_rows, sl = cache[key]
            oracle.sgmv_rows(rows, x_rows, sl, p["lora_ids"], p["grouped_offsets"], p["end"], p["in_dim"],
                             p["R"], p["S"], parallel=parallel)
        return rows.size

    return run, end


def _time_oracle(run, end, parallel, budget_s):
    """Routed rows per second of one oracle build on a bounded sample."""
    probe = min(end, 64 if parallel else 8)
    run(probe, parallel)  # warm (builds/loads the oracle, converts rows)
    t0 = time.perf_counter()
    run(probe, parallel)
    per_row = max((time.perf_counter() - t0) / probe, 1e-7)
    nrows = int(max(1, min(end, budget_s / 3 / per_row)))
    run(nrows, parallel)  # convert
    reps, done, t0 = 0, 0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s and reps < 1000:
        done += run(nrows, parallel)
        reps += 1
    dt = time.perf_counter() - t0
    return done / dt, nrows, reps, dt


def cpu_baseline(workload, budget_s=12.0):
    """The oracle on the host: the OpenMP build on every core of the affinity
    mask (the reported value) and the single-threaded build beside it."""
    import oracle
    from workloads.synthetic import SPECS

    cores = len(os.sched_getaffinity(0))
    run, end = oracle_step_sampler(workload, 0)
    probs = " + ".join(SPECS[workload].problems)
    v1, n1, r1, d1 = _time_oracle(run, end, False, budget_s / 2)
    single = {"value": v1, "unit": "tokens/s", "cores": 1, "kind": "oracle",
              "sample": "first %d of %d routed rows of one %s batch (%s), %d repetitions, %.1f s, "
                        "single-threaded C in double" % (n1, end, workload, probs, r1, d1)}
    model = cpu_model()
    if not oracle.omp_available():
        single["cpu_model"] = model
        single["note"] = "no OpenMP build on this host"
        return single
    threads = oracle.threads(True, cores)
    vp, n_p, rp, dp = _time_oracle(run, end, True, budget_s / 2)
    return {"value": vp, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": "first %d of %d routed rows of one %s batch (%s), %d repetitions, %.1f s, OpenMP build "
                      "of the C oracle (double) over rows on %d threads" % (n_p, end, workload, probs, rp, dp, threads),
            "cpu_model": model, "affinity_cores": cores, "single_thread": single}


def run_reference(args):
    """The reference arm: the CPU oracle (OpenMP build, all cores of the
    affinity mask) timed on a bounded per-step sample of the workload."""
    rank, world, _ = _env_rank()
    if rank != 0:
        return 0
    import oracle
    if args.steps <= 0:
        args.steps = 20
    cores = len(os.sched_getaffinity(0))
    parallel = oracle.omp_available()
    threads = oracle.threads(True, cores) if parallel else 1
    run, end = oracle_step_sampler(args.workload, 0)
    probe = min(end, 64 if parallel else 4)
    run(probe, parallel)
    t0 = time.perf_counter()
    run(probe, parallel)
    per_row = max((time.perf_counter() - t0) / probe, 1e-7)
    steps_total = args.steps + args.warmup
    nrows = int(max(1, min(end, 150.0 / steps_total / per_row)))
    run(nrows, parallel)
    for _ in range(args.warmup):
        run(nrows, parallel)
    t0 = time.perf_counter()
    done = 0
    for _ in range(args.steps):
        done += run(nrows, parallel)
    dt = time.perf_counter() - t0
    val = done / dt
    kind = ("OpenMP build of the C oracle (double) on %d threads" % threads) if parallel else \
        "single-threaded C oracle (double)"
    out = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "config": {"workload": args.workload, "desc": WORKLOAD_DESC[args.workload]},
           "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                            "sample": "first %d of %d routed rows per step (%s), %s"
                                      % (nrows, end, " + ".join(_spec_problems(args.workload)), kind),
                            "cpu_model": cpu_model()},
           "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))
    return 0


def _spec_problems(workload):
    from workloads.synthetic import SPECS
    return SPECS[workload].problems


# -------------------------------------------------------------- GPU arm --

class WorkloadBench:
    """Input sets, pre-marshalled calls and CUDA graphs of one workload."""

    def __init__(self, name, args, rank, lk, torch, stream, l2, max_sets=64):
        from workloads import device, synthetic as sy
        self.name, self.torch, self.stream, self.lk = name, torch, stream, lk
        spec = sy.SPECS[name]
        self.P0, self.P1 = spec.problems
        sets, foot = [], 0
        # Input sets are the layers of one batch: each has its own x, y and
        # adapter stacks, and (as in one decode step) all share the batch's
        # routing triple, built and uploaded once.
        while len(sets) < max_sets:
            share = bool(sets)
            raw = sy.draw(spec, rank_seed(rank, len(sets)),
                          requests=(sets[0]["raw"]["req_slot"], sets[0]["raw"]["req_len"]) if share else None)
            shared = (sets[0]["p0"]["route_host"], sets[0]["p0"]["routing"]) if share else None
            d0 = device.prepare(raw, self.P0, fused=spec.fused_qkv, slot_ranks=args.slot_ranks,
                                shared_routing=shared, host_ids=args.routing == "host")
            d1 = device.prepare(raw, self.P1, slot_ranks=args.slot_ranks,
                                shared_routing=(d0["route_host"], d0["routing"]))
            b0 = algorithmic_bytes(d0["route_host"], raw, self.P0, slot_ranks=args.slot_ranks)
            b1 = algorithmic_bytes(d1["route_host"], raw, self.P1, slot_ranks=args.slot_ranks)
            sets.append({"raw": raw, "p0": d0, "p1": d1, "bytes": b0 + b1, "b0": b0, "b1": b1,
                         "f0": algorithmic_flops(d0["route_host"], raw, self.P0), "E": d0["route_host"]["end"]})
            foot += b0 + b1
            if foot >= 4 * l2 and len(sets) >= 2:
                break
        self.sets, self.NS, self.foot = sets, len(sets), foot
        for s in sets:
            s["call0"] = lk.CallBuilder(s["p0"]["problem"], s["p0"]["routing"], s["p0"]["workspace"])
            s["call1"] = lk.CallBuilder(s["p1"]["problem"], s["p1"]["routing"], s["p1"]["workspace"])
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):  # eager warm (first-launch attribute setup)
            for s in sets:
                s["call0"].apply(stream)
                s["call1"].apply(stream)
        stream.synchronize()
        self.launches_per_step = sets[0]["call0"].last_launches + sets[0]["call1"].last_launches
        self.path_bits = (sets[0]["call0"].last_path, sets[0]["call1"].last_path)
        self.g_all = self._graph(lambda st: [self._step(i, st) for i in range(self.NS)])
        self.g_p0 = self._graph(lambda st: [s["call0"].apply(st) for s in sets])
        self.g_p1 = self._graph(lambda st: [s["call1"].apply(st) for s in sets])
        self.nwarm = 20  # set 0's first-problem apply, back to back: inputs stay in L2
        self.g_warm = self._graph(lambda st: [sets[0]["call0"].apply(st) for _ in range(self.nwarm)])
        self.g_rem = {}

    def _step(self, i, st):
        s = self.sets[i % self.NS]
        s["call0"].apply(st)
        s["call1"].apply(st)

    def _graph(self, body):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            body(torch.cuda.current_stream())
        return g

    def prepare_steps(self, k):
        """Capture (outside any timed region) the graph of k mod NS steps."""
        r = k % self.NS
        if r and r not in self.g_rem:
            self.g_rem[r] = self._graph(lambda st: [self._step(i, st) for i in range(r)])

    def run_steps(self, k):
        """k steps over sets 0, 1, ..., from multi-step graphs (k // NS replays
        of the all-sets graph, then one graph of the remaining steps)."""
        for _ in range(k // self.NS):
            self.g_all.replay()
        r = k % self.NS
        if r:
            self.g_rem[r].replay()

    def steps_tokens_bytes(self, k):
        return (sum(self.sets[i % self.NS]["E"] for i in range(k)),
                sum(self.sets[i % self.NS]["bytes"] for i in range(k)))

    def trials(self, graph, units, min_ms=30.0, n=5, sampler=None):
        """n trials, each replaying `graph` (units apply/step units per replay)
        enough times to last >= min_ms; per-unit ms of each trial."""
        torch, st = self.torch, self.stream
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(st):
            graph.replay()
            e0.record(st)
            graph.replay()
            e1.record(st)
        torch.cuda.synchronize()
        one = max(e0.elapsed_time(e1), 1e-3)
        reps = int(max(1, min(100000, min_ms / one)))
        out = []
        for _ in range(n):
            w0 = time.time()
            with torch.cuda.stream(st):
                e0.record(st)
                for _ in range(reps):
                    graph.replay()
                e1.record(st)
            torch.cuda.synchronize()
            if sampler:
                sampler.mark(w0, time.time())
            out.append(e0.elapsed_time(e1) / (reps * units))
        return out


def roofline_block(wb, trials_ms, peak, peak_kind, tpeak, tpeak_kind, traffic=None):
    med = statistics.median(trials_ms)
    qbytes = statistics.mean(s["b0"] for s in wb.sets)
    qflops = statistics.mean(s["f0"] for s in wb.sets)
    achieved = qbytes / (med * 1e-3) / 1e9
    multi = len(_names(wb.P0)) > 1
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "kernel": "%s SGMV apply (shrink + expand)" % (("fused-" + wb.P0) if multi else wb.P0),
            "peak_source": ("%s HBM copy bandwidth (MEASURED_PEAKS.json)" % peak_kind) if peak_kind == "measured"
            else "fallback 6.8 TB/s",
            "algorithmic_bytes_per_launch": int(qbytes), "avg_launch_us": round(med * 1e3, 3),
            "trials_us": [round(t * 1e3, 3) for t in trials_ms],
            "spread_us": round((max(trials_ms) - min(trials_ms)) * 1e3, 3),
            "flops_per_launch": int(qflops),
            "t_hbm_us": round(qbytes / (peak * 1e9) * 1e6, 3),
            "t_tensor_us": round(qflops / (tpeak * 1e12) * 1e6, 3),
            "tensor_peak_tflops": tpeak,
            "tensor_peak_source": ("%s bf16 dense (MEASURED_PEAKS.json)" % tpeak_kind) if tpeak_kind == "measured"
            else "fallback 1.9 PFLOP/s"}


def _profiled_traffic(workload):
    """DRAM bytes per fused-qkv apply from the committed ncu summary, if present
    and taken on the kernels as they are now."""
    path = os.path.join(ROOT, "profiles", "traffic_%s.json" % workload)
    if os.path.exists(path):
        try:
            d = json.load(open(path))
        except (OSError, ValueError):
            return None
        if d.get("stale"):
            return None
        return d.get("dram_bytes_per_qkv_apply")
    return None


def unsorted_block(wb, sampler, peaks):
    """The first problem's apply on the same batch given in ARRIVAL order:
    x and y rows as the requests arrived, token_rows (lora_build_token_rows)
    mapping the sorted positions to them (the per-token routing of the vLLM
    page, section 6), timed like the sorted apply."""
    lk, torch = wb.lk, wb.torch
    calls = []
    for s in wb.sets:
        d = s["p0"]
        r, rt, raw = d["routing"], d["route_host"], s["raw"]
        rows = lk.lora_build_token_rows(raw["req_len"], rt["perm"], rt["end"])
        tr = torch.from_numpy(rows).to("cuda")
        s["_token_rows"] = tr
        calls.append(lk.CallBuilder(d["problem"], lk.Routing(r.lora_ids, r.grouped_offsets, r.num_groups, r.end, tr,
                                                             r.host_grouped_offsets, r.host_lora_ids),
                                    d["workspace"]))
    with torch.cuda.stream(wb.stream):
        calls[0].apply(wb.stream)
    wb.stream.synchronize()
    g = wb._graph(lambda st: [c.apply(st) for c in calls])
    t = statistics.median(wb.trials(g, wb.NS, sampler=sampler))
    rb = roofline_block(wb, [t], *peaks, traffic=None)
    return {"avg_apply_us": rb["avg_launch_us"], "frac": rb["frac"], "achieved_GBps": rb["achieved"],
            "kernel_path": hex(calls[0].last_path),
            "note": "same batch with rows in arrival order and token_rows: x rows gathered by the shrink, y rows "
                    "read and written in place by the expand"}


def device_routing_block(wb, sampler, peaks):
    """The first problem's apply with the routing's device arrays only (no
    host copies: no tile table for the mma.sync shrink, one kernel family for
    the whole call), for comparison with the default host-copy routing."""
    lk = wb.lk
    calls = []
    for s in wb.sets:
        d = s["p0"]
        r = d["routing"]
        calls.append(lk.CallBuilder(d["problem"], lk.Routing(r.lora_ids, r.grouped_offsets, r.num_groups, r.end),
                                    d["workspace"]))
    with wb.torch.cuda.stream(wb.stream):
        calls[0].apply(wb.stream)
    wb.stream.synchronize()
    g = wb._graph(lambda st: [c.apply(st) for c in calls])
    t = statistics.median(wb.trials(g, wb.NS, sampler=sampler))
    rb = roofline_block(wb, [t], *peaks, traffic=None)
    return {"avg_apply_us": rb["avg_launch_us"], "frac": rb["frac"], "kernel_path": hex(calls[0].last_path),
            "note": "routing without host copies (device lora_ids / grouped_offsets only)"}


def workload_summary(wb, sampler, peaks):
    """Secondary block: step and per-projection times, roofline of the first
    problem's apply (median of 5 trials), warm-L2 time."""
    peak, peak_kind, tpeak, tpeak_kind = peaks
    step_ms = wb.trials(wb.g_all, wb.NS, sampler=sampler)
    q_ms = wb.trials(wb.g_p0, wb.NS, sampler=sampler)
    o_ms = wb.trials(wb.g_p1, wb.NS, sampler=sampler)
    w_ms = wb.trials(wb.g_warm, wb.nwarm, min_ms=10.0, n=3)
    med_step = statistics.median(step_ms)
    tokens = statistics.mean(s["E"] for s in wb.sets)
    ob = statistics.mean(s["b1"] for s in wb.sets)
    med_o = statistics.median(o_ms)
    med_w = statistics.median(w_ms)
    return {
        "desc": WORKLOAD_DESC[wb.name],
        "tokens_per_s": round(tokens / (med_step * 1e-3), 1), "routed_tokens_per_step": tokens,
        "ms_per_step": round(med_step, 5), "step_trials_us": [round(t * 1e3, 3) for t in step_ms],
        "input_sets": wb.NS, "footprint_MB": round(wb.foot / 1e6, 1),
        "roofline": roofline_block(wb, q_ms, peak, peak_kind, tpeak, tpeak_kind, _profiled_traffic(wb.name)),
        "per_projection": {
            wb.P0: {"avg_apply_us": round(statistics.median(q_ms) * 1e3, 3),
                    "GBps": round(statistics.mean(s["b0"] for s in wb.sets) / (statistics.median(q_ms) * 1e-3) / 1e9,
                                  1)},
            wb.P1: {"avg_apply_us": round(med_o * 1e3, 3), "GBps": round(ob / (med_o * 1e-3) / 1e9, 1)}},
        "warm_l2": {"avg_apply_us": round(med_w * 1e3, 3),
                    "GBps": round(wb.sets[0]["b0"] / (med_w * 1e-3) / 1e9, 1),
                    "note": "%s apply of input set 0, %d back to back per graph replay: inputs in L2, not an HBM "
                            "number" % (wb.P0, wb.nwarm)},
        "kernel_paths": [hex(b) for b in wb.path_bits], "launches_per_step": wb.launches_per_step,
    }


def base_fused_block(wb, sampler, peaks):
    """The delta fused into the base projection (lora_base_gemm_apply) against
    the base GEMM (cuBLAS through torch.matmul, the library comparison) plus
    lora_sgmv_apply, on the first problem of every input set; synthetic base
    weights W0 ~ N(0, 1/in)."""
    torch, lk, st = wb.torch, wb.lk, wb.stream
    peak = peaks[0]
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1234)
    items = []
    for s in wb.sets:
        d = s["p0"]
        x, y = d["x"], d["y_all"]
        O, k = y.shape[1], x.shape[1]
        W0 = (torch.randn((O, k), device="cuda", generator=gen, dtype=torch.float32) / k ** 0.5).to(torch.bfloat16)
        offs = np.cumsum([0] + d["outs"])[:-1]
        base = [(W0, int(o) * k, k) for o in offs]
        items.append((d, x, y, W0, base))
    torch.cuda.synchronize()

    def fused(cs):
        for d, x, y, W0, base in items:
            lk.lora_base_gemm_apply(d["problem"], d["routing"], base, d["workspace"], cs)

    def separate(cs):
        for (d, x, y, W0, base), s in zip(items, wb.sets):
            torch.matmul(x, W0.t(), out=y)
            s["call0"].apply(cs)

    with torch.cuda.stream(st):
        fused(st)
        path_bits = lk.lora_last_call_path()[0]
        separate(st)
    st.synchronize()
    g_f, g_s = wb._graph(fused), wb._graph(separate)
    tf = statistics.median(wb.trials(g_f, wb.NS, sampler=sampler))
    ts = statistics.median(wb.trials(g_s, wb.NS, sampler=sampler))
    d0 = wb.sets[0]["p0"]
    T, k = d0["x"].shape
    O = d0["y_all"].shape[1]
    lora = statistics.mean(s["b0"] for s in wb.sets)
    E = statistics.mean(s["E"] for s in wb.sets)
    e = 2
    bytes_fused = T * k * e + O * k * e + T * O * e + (lora - E * k * e - 2 * E * O * e)
    bytes_sep = (T * k * e + O * k * e + T * O * e) + lora
    return {"unit": "%s projection of one layer: every row's W0 x plus the delta on routed rows" % wb.P0,
            "fused_us": round(tf * 1e3, 3), "separate_us": round(ts * 1e3, 3),
            "separate_desc": "torch.matmul (cuBLAS) base GEMM into y, then lora_sgmv_apply",
            "fused_bytes": int(bytes_fused), "separate_bytes": int(bytes_sep),
            "fused_GBps": round(bytes_fused / (tf * 1e-3) / 1e9, 1),
            "fused_frac_of_hbm": round(bytes_fused / (tf * 1e-3) / 1e9 / peak, 4),
            "fused_tflops": round(2.0 * T * O * k / (tf * 1e-3) / 1e12, 1),
            "kernel_path": hex(path_bits)}


def spawn_replicas(args):
    """--gpus N > 1 without a launcher: start N ranks with torch.distributed.run."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(args.gpus),
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.run(cmd).returncode


def run_ours(args):
    import torch

    rank, world, local = _env_rank()
    if args.gpus > 1 and world == 1:
        return spawn_replicas(args)
    if world > 1 and args.gpus != world:
        raise SystemExit("--gpus %d but WORLD_SIZE=%d" % (args.gpus, world))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev_idx = torch.cuda.current_device()
    import __graft_entry__ as ge
    ge.build()
    import adapter_sgmv_lora_gb300 as lk

    props = torch.cuda.get_device_properties(dev_idx)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20) or 126 * 2 ** 20)
    stream = torch.cuda.Stream()
    peak, peak_kind = _peaks()
    tpeak, tpeak_kind = _tensor_peak()
    peaks = (peak, peak_kind, tpeak, tpeak_kind)

    wb = WorkloadBench(args.workload, args, rank, lk, torch, stream, l2, max_sets=args.sets or 64)
    NS = wb.NS
    nwarm = max(args.warmup, 3)
    wb.prepare_steps(nwarm)
    with torch.cuda.stream(stream):
        wb.run_steps(nwarm)
    stream.synchronize()

    if args.steps <= 0:
        # Default: about one second of timed work (at least 640 steps).
        per = statistics.median(wb.trials(wb.g_all, NS, min_ms=20.0, n=3))
        k = int(min(200000, max(640, 1000.0 / max(per, 1e-4))))
        if dist:
            kt = torch.tensor([k], device="cuda")
            dist.all_reduce(kt, op=dist.ReduceOp.MAX)
            k = int(kt.item())
        args.steps = k
    wb.prepare_steps(args.steps)
    with torch.cuda.stream(stream):  # the timed steps' graphs once more, untimed
        wb.run_steps(nwarm)
        wb.run_steps(args.steps % NS)
    stream.synchronize()

    # ---- timed region: exactly K steps
    sampler = ClockSampler(dev_idx) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        wb.run_steps(args.steps)
        ev1.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark(wall0, time.time())
    if dist:
        dist.barrier()
    ms = ev0.elapsed_time(ev1)
    tokens, bytes_steps = wb.steps_tokens_bytes(args.steps)

    # ---- roofline and per-projection figures of the main workload
    main = workload_summary(wb, sampler, peaks)
    if args.routing == "host":
        main["device_routing"] = device_routing_block(wb, sampler, peaks)
    (ms,), (tokens,) = reduce_across_ranks([ms], [tokens], dist, "cuda")

    # ---- e2e through the public API with host buffers
    e2e = run_e2e(args, wb.sets, lk, torch, stream, dist)

    # ---- secondary workloads (rank 0 of N=1 runs only: the scaling run times the main one)
    secondary = {}
    if not args.no_secondary and world == 1:
        for name in SECONDARY:
            if name == args.workload:
                continue
            sb = WorkloadBench(name, args, rank, lk, torch, stream, l2)
            secondary[name] = workload_summary(sb, sampler, peaks)
            if args.routing == "host":
                secondary[name]["device_routing"] = device_routing_block(sb, sampler, peaks)
            if name == "prefill8b":
                secondary[name]["unsorted"] = unsorted_block(sb, sampler, peaks)
            if not args.no_base_fused:
                secondary[name]["base_fused"] = base_fused_block(sb, sampler, peaks)
            del sb
            torch.cuda.empty_cache()
    clocks = sampler.stop() if sampler else None

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0
    cfg = {"workload": args.workload, "desc": WORKLOAD_DESC[args.workload], "input_sets": NS,
           "footprint_MB": round(wb.foot / 1e6, 1), "l2_MB": round(l2 / 2 ** 20, 1),
           "l2_policy": "inputs larger than L2: %d rotated input sets, %.0f MB > 4x L2" % (NS, wb.foot / 1e6),
           "routing": "one batch: the input sets are its layers (own x, y, A/B each) sharing one routing triple"
                      + ("; the routing carries host copies of grouped_offsets and lora_ids" if args.routing == "host"
                         else "; device arrays only"),
           "parallelism": "replicas" if world > 1 else "single GPU",
           "slot_ranks": "true ranks passed (A/B bytes counted at ceil16(rank))" if args.slot_ranks
           else "padded to max_lora_rank",
           "timing": "K steps from multi-step CUDA graphs: %d replays of a %d-step graph + one %d-step graph"
                     % (args.steps // NS, NS, args.steps % NS),
           "hbm_GBps_step": round(bytes_steps / (ms * 1e-3) / 1e9, 1),
           "routed_tokens_per_step": tokens / args.steps / max(world, 1)}
    out = {
        "metric": METRIC, "value": tokens / (ms * 1e-3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; random adapters, activations and base outputs)",
        "config": cfg,
        "roofline": main["roofline"],
        "per_projection": main["per_projection"],
        "step_trials": {"ms_per_step_median": main["ms_per_step"], "trials_us": main["step_trials_us"],
                        "note": "5 trials of >= 30 ms of the same steps, for comparison with the K-step region"},
        "warm_l2": main["warm_l2"],
        "kernel_paths": main["kernel_paths"],
        "device_routing": main.get("device_routing"),
        "secondary": secondary,
        "e2e": e2e,
        "gpu_launches": wb.launches_per_step * args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.workload, budget_s=args.cpu_budget)
    print(json.dumps(out))
    if dist:
        dist.destroy_process_group()
    return 0


def run_e2e(args, sets, lk, torch, stream, dist):
    """Host buffers -> device -> apply (both problems) -> host, through the Python API.

    Each input set owns one pinned host buffer laid out x0 | x1 | lora_ids |
    grouped_offsets | y0 | y1 (256-byte aligned regions) and one device buffer
    of the same layout; the two problems and the routing are built over views
    of the device buffer.  Per step: the host routing build (lora_build_routing
    writing the triple straight into the pinned buffer), one pinned H2D of the
    whole buffer on a copy stream, the two lora_sgmv_apply calls
    (pre-marshalled CallBuilders given the step's num_groups / end) on the
    compute stream, one D2H of y0 | y1 on a second copy stream.  Consecutive
    steps use different sets, so one step's copies overlap another's kernels."""
    import dataclasses
    n = min(len(sets), max(4, min(args.steps, 32)))
    up, down = torch.cuda.Stream(), torch.cuda.Stream()

    def align(v):
        return (v + 255) // 256 * 256

    host = []
    for s in sets[:n]:
        raw = s["raw"]
        P0, P1 = raw["problems"]
        S = raw["max_num_loras"]
        parts = [("x0", raw["x_" + P0]), ("x1", raw["x_" + P1]),
                 ("ids", np.zeros(S, np.int32)), ("offs", np.zeros(S + 1, np.int32)),
                 ("y0", raw["y_" + P0]), ("y1", raw["y_" + P1])]
        off, lay = 0, {}
        for name, arr in parts:
            lay[name] = (off, arr.nbytes)
            off = align(off + arr.nbytes)
        total = off
        H = torch.empty(total, dtype=torch.uint8).pin_memory()
        D = torch.empty(total, dtype=torch.uint8, device="cuda")
        for name, arr in parts:
            o, nb = lay[name]
            H[o:o + nb].copy_(torch.from_numpy(np.ascontiguousarray(arr).view(np.uint8).reshape(-1)))
        y_lo = lay["y0"][0]
        y_hi = lay["y1"][0] + lay["y1"][1]

        def dview(name, shape, dtype):
            o, nb = lay[name]
            return D[o:o + nb].view(dtype).view(shape)

        ids_d = dview("ids", (S,), torch.int32)
        offs_d = dview("offs", (S + 1,), torch.int32)
        h = {"H": H, "D": D, "Dy": D[y_lo:y_hi], "out": torch.empty(y_hi - y_lo, dtype=torch.uint8).pin_memory(),
             "ids_np": H[lay["ids"][0]:lay["ids"][0] + 4 * S].view(torch.int32).numpy(),
             "offs_np": H[lay["offs"][0]:lay["offs"][0] + 4 * (S + 1)].view(torch.int32).numpy(),
             "in": torch.cuda.Event(), "out_ev": torch.cuda.Event(), "done": torch.cuda.Event(),
             "h2d": total, "d2h": y_hi - y_lo, "raw": raw, "calls": []}
        h["done"].record()
        for key, xn, yn in (("p0", "x0", "y0"), ("p1", "x1", "y1")):
            d = s[key]
            assert not d["separate_y"], "one y tensor per problem"
            x_v = dview(xn, tuple(d["x"].shape), d["x"].dtype)
            y_v = dview(yn, tuple(d["y_all"].shape), d["y_all"].dtype)
            prob = d["problem"]
            slices = [dataclasses.replace(sl, y=y_v) for sl in prob.slices]
            prob_v = dataclasses.replace(prob, x=x_v, slices=slices)
            # the host copies are the pinned buffer the step's routing build writes
            hc = args.routing == "host"
            routing_v = lk.Routing(ids_d, offs_d, d["routing"].num_groups, d["routing"].end, None,
                                   h["offs_np"] if hc else None, h["ids_np"] if hc else None)
            h["calls"].append(lk.CallBuilder(prob_v, routing_v, d["workspace"]))
        host.append(h)

    moved = {"h2d": 0, "d2h": 0}

    def one(i, st):
        h = host[i]
        raw = h["raw"]
        moved["h2d"] += h["h2d"]
        moved["d2h"] += h["d2h"]
        h["done"].synchronize()  # this set's previous copies and applies have finished
        rt = lk.lora_build_routing(raw["req_slot"], raw["req_len"], raw["max_num_loras"],
                                   out_ids=h["ids_np"], out_offsets=h["offs_np"])
        with torch.cuda.stream(up):
            h["D"].copy_(h["H"], non_blocking=True)
            h["in"].record(up)
        st.wait_event(h["in"])
        for call in h["calls"]:
            call.set_routing(rt["num_groups"], rt["end"])
            call.apply(st)
        h["out_ev"].record(st)
        down.wait_event(h["out_ev"])
        with torch.cuda.stream(down):
            h["out"].copy_(h["Dy"], non_blocking=True)
            h["done"].record(down)
        return rt["end"]

    for i in range(n):
        one(i, stream)
    torch.cuda.synchronize()
    # At least 64 steps, so the copy/compute pipeline reaches its steady
    # state whatever K the value region used (at K = 20 five steps would be
    # mostly fill and drain).
    k = max(min(args.steps // 4, 400), 64, n)
    moved["h2d"] = moved["d2h"] = 0
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    toks = 0
    e0.record(stream)
    up.wait_event(e0)
    last = None
    for i in range(k):
        toks += one(i % n, stream)
        last = host[i % n]
    stream.wait_event(last["done"])
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    (ms,), (toks,) = reduce_across_ranks([ms], [toks], dist, "cuda")
    return {"value": toks / (ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": moved["h2d"] // k,
            "d2h_bytes_per_step": moved["d2h"] // k, "steps": k,
            "note": "per step: host routing build into the pinned input buffer, one pinned H2D of x, y "
                    "(both problems) and the triple, two lora_sgmv_apply calls, one D2H of both y; "
                    "copies on their own streams, overlapping other steps' kernels"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0,
                    help="timed steps (0: about one second of work, at least 640)")
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=MAIN_WORKLOAD, choices=sorted(WORKLOAD_DESC))
    ap.add_argument("--sets", type=int, default=0, help="input sets to rotate (0: enough for 4x L2)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true", help="skip the decode8b / prefill8b blocks")
    ap.add_argument("--no-base-fused", action="store_true",
                    help="skip the delta-in-base-GEMM comparison in the secondary blocks")
    ap.add_argument("--slot-ranks", action="store_true",
                    help="pass the adapters' true ranks so the kernels skip the rank padding")
    ap.add_argument("--cpu-budget", type=float, default=16.0)
    ap.add_argument("--routing", default="host", choices=["host", "device"],
                    help="host: the routing carries host copies of grouped_offsets and lora_ids (as built by "
                         "lora_build_routing; kernels picked per group in mixed batches, a tile table for the "
                         "mma.sync shrink); device: the device arrays only")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
