"""Benchmark: proportional PER sampling on GB300.

One step = one PER "train call" of the minibatch workload: N=262144 fp32
priorities |N(0,1)|+1e-6, alpha=0.6, 32 rounds of
  update the 8192 items sampled in the previous round with new
  |N(0,1)|+1e-6 priorities -> build_cdf -> sample 8192 stratified with
  their IS weights (beta=0.4)
through the library's C ABI, one per_step call per round (one cooperative
launch: update, rebuild, sample and weights with grid barriers between).  value = sampled transitions per second over
all ranks (device-resident inputs); e2e = the same with each step's new
priorities copied in from pinned host memory and the step's indices and
weights copied back, inside the timed region.

--impl reference times the CPU oracle (serial C, fp64) on the same workload
on this host's cores.  With torchrun, every rank runs an independent replica
("replicas only": the method has no exchange step); rank 0 prints one JSON
line.
"""
from __future__ import annotations

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

import workloads  # noqa: E402

W = workloads.MINIBATCH
N, B, ROUNDS, ALPHA, BETA = W["N"], W["B"], W["rounds"], W["alpha"], W["beta"]
METRIC = "PER samples/sec (minibatch: build_cdf + sample + IS weights + update, 32 rounds/step)"
UNIT = "samples/s"
WORKLOAD = (f"minibatch N={N} fp32 |N(0,1)|+1e-6, alpha={ALPHA}, {ROUNDS} rounds x "
            f"(build_cdf, sample {B} stratified, IS weights beta={BETA}, update {B} at sampled indices)")
L2_FLUSH_BYTES = 512 << 20

# algorithmic bytes per launch: what each kernel must read and write at least
KERNEL_BYTES = {
    "build_cdf": lambda: 8 * N,                          # 4 B read + 4 B write per item
    "sample_is_weights": lambda: 4 * N + 12 * B,         # CDF windows once; index, p gather, weight
    "update": lambda: 8 * B + 4 * B + 8 * B,             # idx + p read, priority write, winner slot
}
# Per key, the radix sort's four passes: pass 0 reads the priorities twice
# (histogram, scatter) and writes keys and values (16 B); passes 1 and 2 read
# the keys twice and the values once and write both (20 B each); pass 3 reads
# the same and writes the order and its inverse (20 B).
RANK_SORT_BYTES_PER_KEY = 16 + 20 + 20 + 20
KERNEL_BYTES["step"] = lambda: sum(KERNEL_BYTES[k]() for k in ("update", "build_cdf", "sample_is_weights"))


def env_rank():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def rank_seed(rank):
    """Workload seed of one replica: every rank draws its own buffer."""
    return W["seed"] + 1000 * rank


def max_over_ranks(x, dist=None, device="cpu"):
    """The largest value of x over the ranks of the default process group
    (x itself without one): the job's time is its slowest replica's."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(steps, world, t_ms):
    """Samples per second of the whole job: every rank's samples over the
    slowest rank's time."""
    return steps * ROUNDS * B * world / (t_ms / 1e3)


def config_dict(n_gpus):
    return {"workload": WORKLOAD, "N": N, "B": B, "rounds_per_step": ROUNDS, "alpha": ALPHA, "beta": BETA,
            "parallelism": f"replicas x{n_gpus}", "l2": "flushed (512 MiB write) between timed steps"}


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------- clocks ----

class ClockSampler:
    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.bus_id = (bus_id or "").lower()
        self.proc = None
        self.path = os.path.join("/tmp", f"per_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                                          "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            t = [x.strip() for x in line.split(",")]
            if len(t) < 10:
                continue
            if self.bus_id and self.bus_id[-12:] not in t[1].lower():
                continue
            rows.append(t)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def mhz(s):
            try:
                return float(s.split()[0])
            except Exception:
                return None
        sm = [mhz(r[2]) for r in rows if mhz(r[2]) is not None]
        mx = [mhz(r[3]) for r in rows if mhz(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------ our arm -------

def run_ours(args, rank, world, local_rank):
    import torch
    import cdf_scan_gb300 as per

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank)
    seed = rank_seed(rank)
    p0 = workloads.minibatch_priorities(seed=seed)
    newp = np.stack([workloads.minibatch_new_priorities(r, seed=seed) for r in range(ROUNDS)])
    d_p0 = torch.from_numpy(p0).to(dev)
    d_newp = torch.from_numpy(newp).to(dev)
    idx = torch.empty((ROUNDS, B), dtype=torch.int32, device=dev)
    wts = torch.empty((ROUNDS, B), dtype=torch.float32, device=dev)
    h_newp = torch.from_numpy(newp).pin_memory()
    h_idx = torch.empty((ROUNDS, B), dtype=torch.int32).pin_memory()
    h_w = torch.empty((ROUNDS, B), dtype=torch.float32).pin_memory()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    ctx = per.PerContext(N, ALPHA, per.PER_SCAN)
    h = ctx.handle
    per.per_set_priorities(h, d_p0)

    # one step = 32 rounds through the C ABI; captured once as a CUDA graph.
    # Round r applies the updates of the items round r-1 sampled (round 0:
    # the previous step's last round), rebuilds and samples.
    calls = {
        "step": lambda r: per.per_step(h, idx[(r - 1) % ROUNDS], d_newp[(r - 1) % ROUNDS], B, seed, r * B,
                                       per.PER_SCAN, BETA, idx[r], wts[r]),
    }
    # the same work as three calls per round (reported beside the step)
    split_calls = {
        "update": lambda r: per.per_update(h, idx[(r - 1) % ROUNDS], d_newp[(r - 1) % ROUNDS]),
        "build_cdf": lambda r: per.per_build_cdf(h),
        "sample_is_weights": lambda r: per.per_sample_weighted(h, B, seed, r * B, per.PER_SCAN, BETA, idx[r], wts[r]),
    }
    per.per_build_cdf(h)
    per.per_sample_weighted(h, B, seed, (ROUNDS - 1) * B, per.PER_SCAN, BETA, idx[ROUNDS - 1], wts[ROUNDS - 1])

    def step_eager(fns=calls):
        for r in range(ROUNDS):
            for fn in fns.values():
                fn(r)

    def capture(body):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        before = per.per_launch_count()
        with torch.cuda.graph(g, stream=s):
            body()
        torch.cuda.synchronize()
        return g, per.per_launch_count() - before

    for _ in range(max(args.warmup, 1)):
        step_eager()  # also configures every kernel before capture
        step_eager(split_calls)
    torch.cuda.synchronize()
    step_graph, kernels_per_step = capture(step_eager)
    split_graph, _ = capture(lambda: step_eager(split_calls))
    kind_graphs = {k: capture(lambda fn=fn: [fn(r) for r in range(ROUNDS)])[0]
                   for k, fn in {**calls, **split_calls}.items()}
    stream = torch.cuda.current_stream()

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
            torch.cuda.synchronize()

    def timed(steps, graph, e2e=False):
        total_ms = 0.0
        for _ in range(steps):
            flush.zero_()
            barrier()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            if e2e:
                d_newp.copy_(h_newp, non_blocking=True)
            graph.replay()
            if e2e:
                h_idx.copy_(idx, non_blocking=True)
                h_w.copy_(wts, non_blocking=True)
            b.record(stream)
            b.synchronize()
            total_ms += a.elapsed_time(b)
        barrier()
        return total_ms

    for _ in range(args.warmup):
        step_graph.replay()
    barrier()
    props = torch.cuda.get_device_properties(dev)
    clocks = ClockSampler(getattr(props, "pci_bus_id", None))
    clocks.start()
    t_ms = timed(args.steps, step_graph)
    clk = clocks.stop()
    e2e_ms = timed(args.steps, step_graph, e2e=True)
    # per-kernel durations: each call kind replayed alone (32 launches per
    # replay, L2 flushed before each replay, as in the step)
    kreps = max(3, min(args.steps, 50))
    per_kernel = {k: timed(kreps, g) / (kreps * ROUNDS) for k, g in kind_graphs.items()}
    split_ms = timed(kreps, split_graph) / kreps
    status = per.per_check(h)
    if status != 0:
        raise RuntimeError(f"device status after timing: {per.per_status_str(status)}")

    t_ms = max_over_ranks(t_ms, dist, dev)
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    result = None
    if rank == 0:
        peak, peak_kind = load_peaks()
        name = "step"  # the one kernel of the timed step
        avg_s = per_kernel[name] / 1e3
        algo = KERNEL_BYTES[name]()
        achieved = algo / avg_s / 1e9
        roofline = {"bound": "hbm", "kernel": name, "achieved": round(achieved, 1), "peak": peak,
                    "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                    "traffic": traffic_for(name), "avg_launch_us": round(avg_s * 1e6, 3),
                    "algorithmic_bytes_per_launch": algo}
        result = {
            "metric": METRIC, "value": job_throughput(args.steps, world, t_ms), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded Philox draws; no dataset)", "config": config_dict(world),
            "e2e": {"value": job_throughput(args.steps, world, e2e_ms), "unit": UNIT,
                    "h2d_bytes_per_step": int(ROUNDS * B * 4),
                    "d2h_bytes_per_step": int(ROUNDS * B * 8)},
            "gpu_launches": int(kernels_per_step * args.steps),
            "roofline": roofline,
            "kernel_us_per_launch": {k: round(v * 1e3, 3) for k, v in per_kernel.items()},
            "us_per_round": round(t_ms / args.steps / ROUNDS * 1e3, 2),
            "split_calls_us_per_round": round(split_ms / ROUNDS * 1e3, 2),
            "clocks": clk,
            "impl": "gb300",
            "notes": "step = one CUDA-graph replay of 32 per_step calls through the C ABI (one cooperative "
                     "launch per round); kernel_us_per_launch also times the three separate calls of the same "
                     "round (update, build_cdf, sample_is_weights) and split_calls_us_per_round the round as "
                     "those three launches; RNG offsets are fixed per captured round while the priority state "
                     "evolves across steps",
        }
        if not args.no_extras:
            result["extras"] = extras(per, torch, dev, peak)
    ctx.close()
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return result


def source_sha(files):
    """sha256 (16 hex digits) over the named files of the CUDA sources."""
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "cdf_scan_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def traffic_for(kernel_name):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel's sources changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[kernel_name]
        if source_sha(e["sources"]) != e["source_sha"]:
            return None
        return e["dram_bytes_per_launch"]
    except Exception:
        return None


def extras(per, torch, dev, peak):
    """Other headline numbers of the metric, measured in the same run (not
    the bench value): the 16M scan against HBM, the 1M-sample sampler, and
    the tree sample+update step at full fill.  Each is a CUDA graph replayed
    between CUDA events on the capturing stream."""
    out = {}
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def graph_of(body):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            body()
        torch.cuda.synchronize()
        return g

    def time_graph(g, reps, flush_l2=True, per_replay=1):
        stream = torch.cuda.current_stream()
        ts = []
        for _ in range(reps):
            if flush_l2:
                flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b) * 1e3 / per_replay)
        return statistics.median(ts)

    S = workloads.STRESS
    n = S["N"]
    ctx = per.PerContext(n, S["alpha"], per.PER_SCAN)
    per.per_set_priorities(ctx.handle, torch.from_numpy(workloads.stress_priorities()).to(dev))
    for _ in range(3):
        per.per_build_cdf(ctx.handle)
    us = time_graph(graph_of(lambda: per.per_build_cdf(ctx.handle)), 30)
    gbs = 8 * n / (us * 1e-6) / 1e9
    idx = torch.empty(S["B"], dtype=torch.int32, device=dev)
    per.per_sample(ctx.handle, S["B"], 1, 0, per.PER_SCAN, idx)
    us_s = time_graph(graph_of(lambda: per.per_sample(ctx.handle, S["B"], 1, 0, per.PER_SCAN, idx)), 20)
    out["stress_build_cdf"] = {"N": n, "us": round(us, 2), "gbs": round(gbs, 1), "frac_of_measured_peak":
                               round(gbs / peak, 4), "frac_of_nominal_8tbs": round(gbs / 8000.0, 4),
                               "l2": "flushed before each rep", "timing": "one-call graph between events"}
    out["stress_sample"] = {"B": S["B"], "us": round(us_s, 2), "samples_per_s": S["B"] / (us_s * 1e-6),
                            "l2": "flushed before each rep"}
    if per.per_check(ctx.handle) != 0:
        out["stress_build_cdf"]["status"] = "device status not clean"
    ctx.close()
    # comparator, context only: the same CDF and sampling with library kernels
    # (torch.cumsum of p**alpha in fp32, torch.searchsorted of the stratified
    # thresholds), timed the same way
    tp = torch.from_numpy(workloads.stress_priorities()).to(dev)
    tcdf = torch.empty_like(tp)
    tu = ((torch.arange(S["B"], device=dev, dtype=torch.float32) + 0.5) / S["B"])
    tidx = torch.empty(S["B"], dtype=torch.int64, device=dev)

    def torch_cdf():
        torch.cumsum(tp.pow(S["alpha"]), 0, out=tcdf)

    def torch_sample():
        torch.searchsorted(tcdf, tu * tcdf[-1], out=tidx)
    torch_cdf()
    us_tc = time_graph(graph_of(torch_cdf), 30)
    us_ts = time_graph(graph_of(torch_sample), 20)
    out["torch_comparator_16M"] = {"build_cdf_us": round(us_tc, 2), "sample_us": round(us_ts, 2),
                                   "note": "torch.cumsum(p**alpha) and torch.searchsorted on the stress input "
                                           "(library kernels); context only", "l2": "flushed before each rep"}

    T = workloads.TREE
    cap = T["capacity"]
    ctx = per.PerContext(cap, T["alpha"], per.PER_TREE)
    p = workloads.lognormal(cap, workloads.rng(T["seed"], 999))
    per.per_set_priorities(ctx.handle, torch.from_numpy(p).to(dev))
    tidx = torch.empty(T["B"], dtype=torch.int32, device=dev)
    upd_idx = []
    upd_p = []
    for s in range(8):
        per.per_sample(ctx.handle, T["B"], 3, s * T["B"], per.PER_TREE, tidx)
        i, q = workloads.tree_update_batch(s, tidx.cpu().numpy())
        upd_idx.append(torch.from_numpy(i).to(dev))
        upd_p.append(torch.from_numpy(q).to(dev))

    def tree_steps():
        for s in range(8):
            per.per_sample(ctx.handle, T["B"], 3, s * T["B"], per.PER_TREE, tidx)
            per.per_update(ctx.handle, upd_idx[s], upd_p[s])
    tree_steps()
    us_t = time_graph(graph_of(tree_steps), 50, flush_l2=False, per_replay=8)
    out["tree_sample_update_step"] = {"capacity": cap, "B": T["B"], "us": round(us_t, 2), "target_us": 20.0,
                                      "l2": "warm (the 4 MiB tree stays resident across steps)",
                                      "timing": "graph of 8 steps between events, per step"}
    if per.per_check(ctx.handle) != 0:
        out["tree_sample_update_step"]["status"] = "device status not clean"

    def iid_steps():  # the same step with i.i.d. thresholds (mode PER_TREE | PER_IID)
        for s in range(8):
            per.per_sample(ctx.handle, T["B"], 3, s * T["B"], per.PER_TREE | per.PER_IID, tidx)
            per.per_update(ctx.handle, upd_idx[s], upd_p[s])
    iid_steps()
    us_i = time_graph(graph_of(iid_steps), 50, flush_l2=False, per_replay=8)
    out["tree_iid_sample_update_step"] = {"capacity": cap, "B": T["B"], "us": round(us_i, 2),
                                          "l2": "warm (the 4 MiB tree stays resident across steps)",
                                          "timing": "graph of 8 steps between events, per step"}
    if per.per_check(ctx.handle) != 0:
        out["tree_iid_sample_update_step"]["status"] = "device status not clean"
    ctx.close()

    R = workloads.RESAMPLE
    logw = torch.from_numpy(workloads.resample_logw()).to(dev)
    ridx = torch.empty((R["rows"], R["P"]), dtype=torch.int32, device=dev)
    per.per_resample(logw, 6, 0, ridx)
    us_r = time_graph(graph_of(lambda: per.per_resample(logw, 6, 0, ridx)), 20)
    rbytes = 8 * R["rows"] * R["P"]
    out["resample"] = {"rows": R["rows"], "P": R["P"], "us": round(us_r, 2),
                       "gbs": round(rbytes / (us_r * 1e-6) / 1e9, 1),
                       "frac_of_measured_peak": round(rbytes / (us_r * 1e-6) / 1e9 / peak, 4),
                       "l2": "flushed before each rep"}
    # the minibatch step that also returns the sampled transitions: rows of
    # 64 floats (256 B) per item, copied inside the step's launch
    Mb = workloads.MINIBATCH
    ctx = per.PerContext(Mb["N"], Mb["alpha"], per.PER_SCAN)
    per.per_set_priorities(ctx.handle, torch.from_numpy(workloads.minibatch_priorities()).to(dev))
    trans = torch.randn((Mb["N"], 64), generator=torch.Generator(device=dev).manual_seed(7), device=dev)
    gi = [torch.empty(Mb["B"], dtype=torch.int32, device=dev) for _ in range(2)]
    gw = torch.empty(Mb["B"], dtype=torch.float32, device=dev)
    grows = torch.empty((Mb["B"], 64), dtype=torch.float32, device=dev)
    gnew = [torch.from_numpy(workloads.minibatch_new_priorities(r)).to(dev) for r in range(8)]
    per.per_build_cdf(ctx.handle)
    per.per_sample(ctx.handle, Mb["B"], Mb["seed"], 0, per.PER_SCAN, gi[0])

    def gather_steps():
        for r in range(8):
            per.per_step_gather(ctx.handle, gi[r & 1], gnew[r], Mb["B"], Mb["seed"], r * Mb["B"], per.PER_SCAN,
                                Mb["beta"], gi[(r + 1) & 1], gw, trans, grows)
    gather_steps()
    us_g = time_graph(graph_of(gather_steps), 30, flush_l2=False, per_replay=8)
    out["step_gather_minibatch_256B"] = {"N": Mb["N"], "B": Mb["B"], "row_bytes": 256, "us": round(us_g, 2),
                                         "l2": "warm (the transitions stay resident across steps)",
                                         "timing": "graph of 8 steps between events, per step"}
    if per.per_check(ctx.handle) != 0:
        out["step_gather_minibatch_256B"]["status"] = "device status not clean"
    ctx.close()

    # rank-based PER on the minibatch workload: per step, update the 8192
    # sampled items, re-sort all 262,144 by priority, sample 8192 ranks with
    # IS weights (per_step, mode PER_RANK)
    Mb = workloads.MINIBATCH
    ctx = per.PerContext(Mb["N"], Mb["alpha"], per.PER_RANK)
    per.per_set_priorities(ctx.handle, torch.from_numpy(workloads.minibatch_priorities()).to(dev))
    per.per_rank_build(ctx.handle)
    ri = [torch.empty(Mb["B"], dtype=torch.int32, device=dev) for _ in range(2)]
    rw = torch.empty(Mb["B"], dtype=torch.float32, device=dev)
    rnew = [torch.from_numpy(workloads.minibatch_new_priorities(r)).to(dev) for r in range(8)]
    per.per_sample(ctx.handle, Mb["B"], Mb["seed"], 0, per.PER_RANK, ri[0])

    def rank_steps():
        for r in range(8):
            per.per_step(ctx.handle, ri[r & 1], rnew[r], Mb["B"], Mb["seed"], r * Mb["B"], per.PER_RANK,
                         Mb["beta"], ri[(r + 1) & 1], rw)
    rank_steps()
    us_k = time_graph(graph_of(rank_steps), 30, flush_l2=False, per_replay=8)
    us_b = time_graph(graph_of(lambda: per.per_rank_build(ctx.handle)), 30, flush_l2=False)
    out["rank_minibatch_step"] = {"N": Mb["N"], "B": Mb["B"], "us": round(us_k, 2), "sort_us": round(us_b, 2),
                                  "l2": "warm (the 1 MiB priorities stay resident across steps)",
                                  "timing": "graph of 8 steps between events, per step"}
    if per.per_check(ctx.handle) != 0:
        out["rank_minibatch_step"]["status"] = "device status not clean"
    ctx.close()
    # the sort at 16M items (L2 flushed): four 8-bit passes, each reading the
    # keys twice and the values once and writing both (pass 0 reads the
    # priorities; the last writes the order and its inverse)
    ctx = per.PerContext(n, S["alpha"], per.PER_RANK)
    per.per_set_priorities(ctx.handle, torch.from_numpy(workloads.stress_priorities()).to(dev))
    per.per_rank_build(ctx.handle)
    us_16 = time_graph(graph_of(lambda: per.per_rank_build(ctx.handle)), 10)
    sort_bytes = RANK_SORT_BYTES_PER_KEY * n
    out["rank_sort_16M"] = {"N": n, "us": round(us_16, 2), "keys_per_s": n / (us_16 * 1e-6),
                            "gbs": round(sort_bytes / (us_16 * 1e-6) / 1e9, 1),
                            "frac_of_measured_peak": round(sort_bytes / (us_16 * 1e-6) / 1e9 / peak, 4),
                            "bytes_per_key": RANK_SORT_BYTES_PER_KEY, "l2": "flushed before each rep"}
    if per.per_check(ctx.handle) != 0:
        out["rank_sort_16M"]["status"] = "device status not clean"
    ctx.close()

    # the whole particle-filter resample step with D = 4 states per particle:
    # indices, gathered states and the reset log-weights in one launch
    D = 4
    state = torch.randn((R["rows"], R["P"], D), generator=torch.Generator(device=dev).manual_seed(6), device=dev)
    out_state = torch.empty_like(state)
    out_lw = torch.empty_like(logw)
    per.per_resample_step(logw, state, 6, 0, ridx, out_state, out_lw)
    us_s = time_graph(graph_of(lambda: per.per_resample_step(logw, state, 6, 0, ridx, out_state, out_lw)), 20)
    sbytes = R["rows"] * R["P"] * (4 + 4 + 4 + 8 * D)  # logw in, idx out, logw out, states in and out
    out["resample_step_d4"] = {"rows": R["rows"], "P": R["P"], "D": D, "us": round(us_s, 2),
                               "gbs": round(sbytes / (us_s * 1e-6) / 1e9, 1),
                               "frac_of_measured_peak": round(sbytes / (us_s * 1e-6) / 1e9 / peak, 4),
                               "l2": "flushed before each rep"}
    return out


# ------------------------------------------------------ kernel cases --------

KERNEL_CASES = ("scan_stress", "scan_minibatch", "sample_stress", "sample_minibatch", "is_weights_minibatch",
                "update_minibatch", "step_minibatch", "tree_step", "resample", "is_weights_heavy",
                "rank_sort_stress", "rank_step_minibatch", "resample_step")


def kernel_case(name, reps):
    """Run one kernel of one workload `reps` times after setup (for ncu
    captures: -k selects the kernel, -s skips the setup launches).  Prints
    "ok" after a clean device status; no timing."""
    import torch
    import cdf_scan_gb300 as per
    from cdf_scan_gb300 import _build
    _build.build()
    dev = torch.device("cuda", 0)
    ctxs = []
    if name in ("scan_stress", "sample_stress"):
        S = workloads.STRESS
        ctx = per.PerContext(S["N"], S["alpha"], per.PER_SCAN)
        per.per_set_priorities(ctx.handle, torch.from_numpy(workloads.stress_priorities()).to(dev))
        idx = torch.empty(S["B"], dtype=torch.int32, device=dev)
        if name == "scan_stress":
            body = lambda: per.per_build_cdf(ctx.handle)  # noqa: E731
        else:
            per.per_build_cdf(ctx.handle)
            body = lambda: per.per_sample(ctx.handle, S["B"], 1, 0, per.PER_SCAN, idx)  # noqa: E731
    elif name in ("scan_minibatch", "sample_minibatch", "is_weights_minibatch", "update_minibatch",
                  "step_minibatch"):
        ctx = per.PerContext(N, ALPHA, per.PER_SCAN)
        per.per_set_priorities(ctx.handle, torch.from_numpy(workloads.minibatch_priorities()).to(dev))
        per.per_build_cdf(ctx.handle)
        idx = torch.empty(B, dtype=torch.int32, device=dev)
        w = torch.empty(B, dtype=torch.float32, device=dev)
        newp = torch.from_numpy(workloads.minibatch_new_priorities(0)).to(dev)
        per.per_sample(ctx.handle, B, W["seed"], 0, per.PER_SCAN, idx)
        idx2 = torch.empty(B, dtype=torch.int32, device=dev)
        body = {"scan_minibatch": lambda: per.per_build_cdf(ctx.handle),
                "sample_minibatch": lambda: per.per_sample(ctx.handle, B, W["seed"], 0, per.PER_SCAN, idx),
                "is_weights_minibatch": lambda: per.per_is_weights(ctx.handle, idx, BETA, w),
                "update_minibatch": lambda: per.per_update(ctx.handle, idx, newp),
                "step_minibatch": lambda: per.per_step(ctx.handle, idx, newp, B, W["seed"], 0, per.PER_SCAN, BETA,
                                                       idx2, w)}[name]
    elif name == "is_weights_heavy":
        Hv = workloads.HEAVY
        ctx = per.PerContext(Hv["N"], Hv["alpha"], per.PER_SCAN)
        per.per_set_priorities(ctx.handle, torch.from_numpy(workloads.heavy_priorities()).to(dev))
        per.per_build_cdf(ctx.handle)
        idx = torch.empty(Hv["B"], dtype=torch.int32, device=dev)
        w = torch.empty(Hv["B"], dtype=torch.float32, device=dev)
        per.per_sample(ctx.handle, Hv["B"], 4, 0, per.PER_SCAN, idx)
        body = lambda: per.per_is_weights(ctx.handle, idx, Hv["betas"][0], w)  # noqa: E731
    elif name == "tree_step":
        T = workloads.TREE
        ctx = per.PerContext(T["capacity"], T["alpha"], per.PER_TREE)
        p = workloads.lognormal(T["capacity"], workloads.rng(T["seed"], 999))
        per.per_set_priorities(ctx.handle, torch.from_numpy(p).to(dev))
        tidx = torch.empty(T["B"], dtype=torch.int32, device=dev)
        per.per_sample(ctx.handle, T["B"], 3, 0, per.PER_TREE, tidx)
        ui, up = workloads.tree_update_batch(0, tidx.cpu().numpy())
        d_ui, d_up = torch.from_numpy(ui).to(dev), torch.from_numpy(up).to(dev)

        def body():
            per.per_sample(ctx.handle, T["B"], 3, 0, per.PER_TREE, tidx)
            per.per_update(ctx.handle, d_ui, d_up)
    elif name == "rank_sort_stress":
        S = workloads.STRESS
        ctx = per.PerContext(S["N"], S["alpha"], per.PER_RANK)
        per.per_set_priorities(ctx.handle, torch.from_numpy(workloads.stress_priorities()).to(dev))
        body = lambda: per.per_rank_build(ctx.handle)  # noqa: E731
    elif name == "rank_step_minibatch":
        ctx = per.PerContext(N, ALPHA, per.PER_RANK)
        per.per_set_priorities(ctx.handle, torch.from_numpy(workloads.minibatch_priorities()).to(dev))
        per.per_rank_build(ctx.handle)
        idx = torch.empty(B, dtype=torch.int32, device=dev)
        idx2 = torch.empty(B, dtype=torch.int32, device=dev)
        w = torch.empty(B, dtype=torch.float32, device=dev)
        newp = torch.from_numpy(workloads.minibatch_new_priorities(0)).to(dev)
        per.per_sample(ctx.handle, B, W["seed"], 0, per.PER_RANK, idx)
        body = lambda: per.per_step(ctx.handle, idx, newp, B, W["seed"], 0, per.PER_RANK, BETA, idx2, w)  # noqa: E731
    elif name in ("resample", "resample_step"):
        R = workloads.RESAMPLE
        logw = torch.from_numpy(workloads.resample_logw()).to(dev)
        out = torch.empty((R["rows"], R["P"]), dtype=torch.int32, device=dev)
        ctx = None
        if name == "resample":
            body = lambda: per.per_resample(logw, 6, 0, out)  # noqa: E731
        else:  # D = 4 states per particle, log-weights reset into a second buffer
            state = torch.randn((R["rows"], R["P"], 4), generator=torch.Generator(device=dev).manual_seed(6),
                                device=dev)
            out_state = torch.empty_like(state)
            out_lw = torch.empty_like(logw)
            body = lambda: per.per_resample_step(logw, state, 6, 0, out, out_state, out_lw)  # noqa: E731
    else:
        raise SystemExit(f"unknown kernel case {name!r}; one of {', '.join(KERNEL_CASES)}")
    if ctx is not None:
        ctxs.append(ctx)
    for _ in range(reps):
        body()
    torch.cuda.synchronize()
    for c in ctxs:
        if per.per_check(c.handle) != 0:
            raise SystemExit("device status not clean")
        c.close()
    print("ok", flush=True)


# -------------------------------------------------------- oracle arms -------

def oracle_step(p, seed, step):
    """One step of the workload on the CPU oracle (serial C, fp64)."""
    import oracle
    prio = p
    for r in range(ROUNDS):
        C = oracle.cdf64(prio, ALPHA)
        idx, _ = oracle.sample_cdf_f64(C, B, seed, (step * ROUNDS + r) * B)
        oracle.is_weights(prio, N, ALPHA, idx, BETA)
        prio = oracle.apply_updates(prio, idx, workloads.minibatch_new_priorities(r, seed=seed))
    return prio


def cpu_baseline(seconds=10.0):
    import oracle
    oracle.build()
    p = workloads.minibatch_priorities()
    t0 = time.perf_counter()
    rounds = 0
    step = 0
    while time.perf_counter() - t0 < seconds:
        p = oracle_step(p, W["seed"], step)
        step += 1
        rounds += ROUNDS
    dt = time.perf_counter() - t0
    return {"value": rounds * B / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{step} full steps ({rounds} rounds) of the minibatch workload, {dt:.1f} s, single thread"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    p = workloads.minibatch_priorities()
    for s in range(args.warmup):
        p = oracle_step(p, W["seed"], s)
    t0 = time.perf_counter()
    for s in range(args.steps):
        p = oracle_step(p, W["seed"], args.warmup + s)
    dt = time.perf_counter() - t0
    value = args.steps * ROUNDS * B / dt
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded Philox draws; no dataset)", "config": config_dict(world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{args.steps} full steps of the minibatch workload, single thread"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--kernel-case", choices=KERNEL_CASES, default=None,
                    help="run one kernel of one workload a few times (for profiler captures) and exit")
    ap.add_argument("--reps", type=int, default=5)
    args = ap.parse_args()
    rank, world, local_rank = env_rank()
    if args.kernel_case:
        kernel_case(args.kernel_case, args.reps)
        return
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        from cdf_scan_gb300 import _build
        if rank == 0 or world == 1:
            _build.build()
        res = run_ours(args, rank, world, local_rank)
        if res is not None and world == 1:
            res["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
