"""Benchmark: proportional PER sampling on GB300.

One step = one PER "train call" of the minibatch workload: N=262144 fp32
priorities |N(0,1)|+1e-6, alpha=0.6, 32 rounds of
  update the 8192 items sampled in the previous round with new
  |N(0,1)|+1e-6 priorities -> build_cdf -> sample 8192 stratified with
  their IS weights (beta=0.4)
through the library's C ABI, one per_step call per round (one cooperative
launch: update, rebuild, sample and weights with grid barriers between).
value = sampled transitions per second over all ranks (device-resident
inputs); e2e = the same with each step's new priorities copied in from pinned
host memory and the step's indices and weights copied back, inside the timed
region.

The JSON line also carries one record per workload of the method (key
"configs": small, minibatch, tree, heavy, stress, resample), each with its
own timings, a roofline for its dominant kernel against the algorithmic
bytes of that workload, the CPU oracle timed on a bounded sample of the same
workload, and the number of sampled indices that differ from the oracle's
search of its own fp64 CDF (only boundary-band differences are possible; the
tests check the band).

L2 is flushed before every timed replay where the record says so: a 512 MiB
buffer is written and then another 512 MiB buffer is read, so that no input
is cached and the flush leaves no dirty lines to be written back inside the
timed region (the 16M scan is also reported after a write-only flush).

--impl reference times the CPU oracle (serial C, fp64) on the same workload
on this host's cores.  With torchrun, every rank runs an independent replica
("replicas only": the method has no exchange step); rank 0 prints one JSON
line.
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

import workloads  # noqa: E402

W = workloads.MINIBATCH
N, B, ROUNDS, ALPHA, BETA = W["N"], W["B"], W["rounds"], W["alpha"], W["beta"]
METRIC = "PER samples/sec (minibatch: build_cdf + sample + IS weights + update, 32 rounds/step)"
UNIT = "samples/s"
WORKLOAD = (f"minibatch N={N} fp32 |N(0,1)|+1e-6, alpha={ALPHA}, {ROUNDS} rounds x "
            f"(build_cdf, sample {B} stratified, IS weights beta={BETA}, update {B} at sampled indices)")
L2_FLUSH_BYTES = 512 << 20

# Algorithmic bytes per launch -- what each kernel must read and write at
# least -- for the minibatch workload's calls.  One fused round (per_step):
# the scan reads p and writes the CDF (8 B per item), each of the B samples
# writes its index and reads at most one 32-byte sector of the CDF, the
# update reads an index and a priority (8 B per sample) and the IS weights
# gather p and write a weight (8 B per sample).
KERNEL_BYTES = {
    "build_cdf": lambda: 8 * N,
    "sample_is_weights": lambda: B * (4 + 32) + 8 * B,
    "update": lambda: 8 * B,
}
KERNEL_BYTES["step"] = lambda: 8 * N + B * (4 + 32) + 8 * B + 8 * B
# Per key, the radix sort's four passes: pass 0 reads the priorities twice
# (histogram, scatter) and writes keys and values (16 B); passes 1 and 2 read
# the keys twice and the values once and write both (20 B each); pass 3 reads
# the same and writes the order and its inverse (20 B).
RANK_SORT_BYTES_PER_KEY = 16 + 20 + 20 + 20


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
            "parallelism": f"replicas x{n_gpus}",
            "l2": "flushed between timed steps (512 MiB write, then 512 MiB read of another buffer)"}


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

class L2Flush:
    """Evicts L2 between timed replays: writes one 512 MiB buffer, then reads
    another (so L2 ends up holding clean lines of neither input); `dirty`
    only writes."""

    def __init__(self, torch, dev):
        self.torch = torch
        self.a = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.b = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.acc = torch.empty((), dtype=torch.float32, device=dev)

    def clean(self):
        self.a.zero_()
        self.torch.sum(self.b, dim=0, out=self.acc)

    def dirty(self):
        self.a.zero_()


def graph_of(torch, body):
    """CUDA graph of body() captured on a side stream."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        body()
    torch.cuda.synchronize()
    return g


def time_graph(torch, g, reps, flush=None, per_replay=1):
    """Median microseconds per body (replay time / per_replay) between CUDA
    events recorded on the replaying stream; flush() before each replay."""
    stream = torch.cuda.current_stream()
    ts = []
    for _ in range(reps):
        if flush is not None:
            flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b) * 1e3 / per_replay)
    return statistics.median(ts)


def roofline(kernel, algo_bytes, us, peak, peak_kind, traffic=None, note=None):
    achieved = algo_bytes / (us * 1e-6) / 1e9
    r = {"bound": "hbm", "kernel": kernel, "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind,
         "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic, "avg_launch_us": round(us, 3),
         "algorithmic_bytes_per_launch": int(algo_bytes)}
    if note:
        r["note"] = note
    return r


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
    flush = L2Flush(torch, dev)
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
        before = per.per_launch_count()
        g = graph_of(torch, body)
        return g, per.per_launch_count() - before

    for _ in range(max(args.warmup, 1)):
        step_eager()  # also configures every kernel before capture
        step_eager(split_calls)
    torch.cuda.synchronize()
    step_graph, kernels_per_step = capture(step_eager)
    split_graph, _ = capture(lambda: step_eager(split_calls))
    kind_graphs = {k: capture(lambda fn=fn: [fn(r) for r in range(ROUNDS)])[0] for k, fn in split_calls.items()}
    stream = torch.cuda.current_stream()

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
            torch.cuda.synchronize()

    def timed(steps, graph, e2e=False):
        total_ms = 0.0
        for _ in range(steps):
            flush.clean()
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
    # the same round as three separate calls, each kind replayed alone (32
    # launches per replay, L2 flushed before each replay), and as a whole
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
        # the roofline kernel's duration from the timed replays themselves: the
        # step is 32 launches of it, so a launch averages ms_per_step / 32
        # (gaps between the graph's launches included: an upper bound)
        step_us = t_ms / args.steps / ROUNDS * 1e3
        rl = roofline("per_step_kernel (update + build_cdf + sample + IS weights, one launch)", KERNEL_BYTES["step"](),
                      step_us, peak, peak_kind, traffic_for("step"),
                      note="latency-bound: the working set (1 MiB of priorities, 1 MiB of CDF) stays in L2")
        result = {
            "metric": METRIC, "value": job_throughput(args.steps, world, t_ms), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded Philox draws; no dataset)", "config": config_dict(world),
            "e2e": {"value": job_throughput(args.steps, world, e2e_ms), "unit": UNIT,
                    "h2d_bytes_per_step": int(ROUNDS * B * 4),
                    "d2h_bytes_per_step": int(ROUNDS * B * 8)},
            "gpu_launches": int(kernels_per_step * args.steps),
            "roofline": rl,
            "kernel_us_per_launch": {"step": round(step_us, 3),
                                     **{k: round(v * 1e3, 3) for k, v in per_kernel.items()}},
            "us_per_round": round(step_us, 2),
            "split_calls_us_per_round": round(split_ms / ROUNDS * 1e3, 2),
            "clocks": clk,
            "impl": "gb300",
            "notes": "step = one CUDA-graph replay of 32 per_step calls through the C ABI (one cooperative "
                     "launch per round); kernel_us_per_launch.step = ms_per_step / 32 from the timed replays; the "
                     "other entries time the three separate calls of the same round (update, build_cdf, "
                     "sample_is_weights), each kind alone, and split_calls_us_per_round the round as those three "
                     "launches; RNG offsets are fixed per captured round while the priority state evolves across "
                     "steps",
        }
    ctx.close()
    if rank == 0 and not args.no_extras:
        result["configs"], result["extras"], checks = measure_configs(per, torch, dev, peak, peak_kind, flush,
                                                                      result)
        if world == 1:
            oracle_legs(result["configs"], checks, args.cpu_seconds)
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


def measure_configs(per, torch, dev, peak, peak_kind, flush, head):
    """One record per workload, measured in this run; returns (configs,
    extras, checks), `checks` holding the GPU results that the oracle legs
    compare with."""
    cfg, checks, extras = {}, {}, {}
    tensor = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731

    # ---- small: N = 8192, B = 1024 (latency-bound: 64 KiB, L2-resident)
    Sm = workloads.SMALL
    n, b = Sm["N"], Sm["B"]
    p = workloads.small_priorities()
    ctx = per.PerContext(n, Sm["alpha"], per.PER_SCAN)
    per.per_set_priorities(ctx.handle, tensor(p))
    i_s = torch.empty(b, dtype=torch.int32, device=dev)
    w_s = torch.empty(b, dtype=torch.float32, device=dev)
    per.per_build_cdf(ctx.handle)
    per.per_sample(ctx.handle, b, Sm["seed"], 0, per.PER_SCAN, i_s)
    checks["small"] = {"p": p, "idx": i_s.cpu().numpy()}
    reps = 32
    us = {
        "build_cdf": time_graph(torch, graph_of(torch, lambda: [per.per_build_cdf(ctx.handle) for _ in range(reps)]),
                                50, per_replay=reps),
        "sample": time_graph(torch, graph_of(torch, lambda: [per.per_sample(ctx.handle, b, Sm["seed"], 0,
                                                                           per.PER_SCAN, i_s) for _ in range(reps)]),
                             50, per_replay=reps),
        "is_weights": time_graph(torch, graph_of(torch, lambda: [per.per_is_weights(ctx.handle, i_s, Sm["beta"], w_s)
                                                                 for _ in range(reps)]), 50, per_replay=reps),
        "combined_three_calls": time_graph(torch, graph_of(torch, lambda: [
            (per.per_build_cdf(ctx.handle), per.per_sample(ctx.handle, b, Sm["seed"], 0, per.PER_SCAN, i_s),
             per.per_is_weights(ctx.handle, i_s, Sm["beta"], w_s)) for _ in range(reps)]), 50, per_replay=reps),
        "combined_per_step": time_graph(torch, graph_of(torch, lambda: [
            per.per_step(ctx.handle, None, None, b, Sm["seed"], 0, per.PER_SCAN, Sm["beta"], i_s, w_s)
            for _ in range(reps)]), 50, per_replay=reps),
    }
    assert per.per_check(ctx.handle) == 0
    ctx.close()
    cfg["small"] = {
        "workload": f"N={n} fp32 |N(0,1)|+1e-6, alpha={Sm['alpha']}, beta={Sm['beta']}, B={b} stratified",
        "us_per_call": {k: round(v, 2) for k, v in us.items()},
        "samples_per_s": b / (us["combined_per_step"] * 1e-6),
        "roofline": roofline("build_cdf_wave_kernel<256>", 8 * n, us["build_cdf"], peak, peak_kind,
                             note="latency-bound: 64 KiB, L2-resident; the pages' point of comparison (PufferLib "
                                  "PR #615 section 1: 90 us serial, 7.5 us two-level, GPU not stated)"),
        "l2": "warm (the 64 KiB buffer stays resident between calls); graph of 32 calls per replay"}

    # ---- minibatch: the headline step (above); its record
    cfg["minibatch"] = {
        "workload": WORKLOAD, "us_per_round": head["us_per_round"],
        "split_calls_us_per_round": head["split_calls_us_per_round"], "samples_per_s": head["value"],
        "ms_per_32_rounds": head["ms_per_step"],
        "vs_serial_scan_on_the_pages": "PufferLib PR #615 section 1: 32 x 2.85 ms of serial build_cdf per train "
                                       "call at B=262144 (GPU not stated)",
        "roofline": head["roofline"], "l2": head["config"]["l2"]}
    ctx = per.PerContext(N, ALPHA, per.PER_SCAN)
    p = workloads.minibatch_priorities()
    per.per_set_priorities(ctx.handle, tensor(p))
    i_m = torch.empty(B, dtype=torch.int32, device=dev)
    w_m = torch.empty(B, dtype=torch.float32, device=dev)
    per.per_step(ctx.handle, None, None, B, W["seed"], 0, per.PER_SCAN, BETA, i_m, w_m)
    checks["minibatch"] = {"p": p, "idx": i_m.cpu().numpy()}
    assert per.per_check(ctx.handle) == 0
    ctx.close()

    # ---- tree: capacity 500,000 (2^19 leaves); the 400-step growth loop
    T = workloads.TREE
    cap, tb = T["capacity"], T["B"]
    ctx = per.PerContext(cap, T["alpha"], per.PER_TREE)
    prio = np.zeros(cap, np.float32)
    init = workloads.tree_initial()
    prio[:init.size] = init
    per.per_set_priorities(ctx.handle, tensor(prio))
    size, head_pos = init.size, init.size % cap
    per.per_set_size(ctx.handle, size)
    out = torch.empty(tb, dtype=torch.int32, device=dev)
    # a first pass draws every step's samples, so that the timed pass can
    # enqueue all 400 steps (insert, sample, update) without host work between
    steps = T["steps"]
    plan = []
    for s in range(steps):
        ins = workloads.tree_insert(s)
        ins_idx = ((head_pos + np.arange(ins.size)) % cap).astype(np.int32)
        per.per_update(ctx.handle, tensor(ins_idx), tensor(ins))
        prio = workloads_apply(prio, ins_idx, ins)
        head_pos = (head_pos + ins.size) % cap
        size = min(size + ins.size, cap)
        per.per_set_size(ctx.handle, size)
        per.per_sample(ctx.handle, tb, T["seed"], s * tb, per.PER_TREE, out)
        ui, up = workloads.tree_update_batch(s, out.cpu().numpy())
        per.per_update(ctx.handle, tensor(ui), tensor(up))
        prio = workloads_apply(prio, ui, up)
        plan.append((tensor(ins_idx), tensor(ins), size, tensor(ui), tensor(up)))
    checks["tree"] = {"prio": prio, "size": size}
    per.per_sample(ctx.handle, tb, T["seed"], steps * tb, per.PER_TREE, out)
    checks["tree"]["idx"] = out.cpu().numpy()
    ctx.close()
    ctx = per.PerContext(cap, T["alpha"], per.PER_TREE)
    prio0 = np.zeros(cap, np.float32)
    prio0[:init.size] = init
    per.per_set_priorities(ctx.handle, tensor(prio0))
    per.per_set_size(ctx.handle, init.size)
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for s, (ii, iv, sz, ui, up) in enumerate(plan):
        ev[s][0].record(stream)
        per.per_update(ctx.handle, ii, iv)
        per.per_set_size(ctx.handle, sz)
        ev[s][1].record(stream)
        per.per_sample(ctx.handle, tb, T["seed"], s * tb, per.PER_TREE, out)
        per.per_update(ctx.handle, ui, up)
        ev[s][2].record(stream)
    torch.cuda.synchronize()
    ins_us = [ev[s][0].elapsed_time(ev[s][1]) * 1e3 for s in range(steps)]
    stp_us = [ev[s][1].elapsed_time(ev[s][2]) * 1e3 for s in range(steps)]
    assert per.per_check(ctx.handle) == 0
    fill_curve = []
    for lo in range(0, steps, 25):
        sl = slice(lo, min(lo + 25, steps))
        fill_curve.append({"steps": f"{lo}-{sl.stop - 1}", "fill": int(plan[sl.stop - 1][2]),
                           "step_us": round(statistics.median(stp_us[sl]), 2),
                           "insert_us": round(statistics.median(ins_us[sl]), 2)})
    # the steady state at full fill: a graph of 8 sample + update steps
    tidx = torch.empty(tb, dtype=torch.int32, device=dev)
    ups = plan[-8:]

    def tree_steps(mode=per.PER_TREE):
        for s in range(8):
            per.per_sample(ctx.handle, tb, T["seed"], s * tb, mode, tidx)
            per.per_update(ctx.handle, ups[s][3], ups[s][4])
    tree_steps()
    us_t = time_graph(torch, graph_of(torch, tree_steps), 50, per_replay=8)
    tree_steps(per.PER_TREE | per.PER_IID)
    us_i = time_graph(torch, graph_of(torch, lambda: tree_steps(per.PER_TREE | per.PER_IID)), 50, per_replay=8)
    assert per.per_check(ctx.handle) == 0
    ctx.close()
    levels = 19
    cfg["tree"] = {
        "workload": f"segment tree capacity {cap} (2^19 leaves, fp32), fill {init.size} -> {cap} by insert_batch of "
                    f"{T['insert']} lognormal(0,1); per step sample {tb}, update {tb} (20% duplicate indices); "
                    f"{steps} steps; alpha={T['alpha']}",
        "sample_update_step_us": round(us_t, 2), "target_us": 20.0,
        "iid_sample_update_step_us": round(us_i, 2),
        "insert_us_median": round(statistics.median(ins_us), 2),
        "step_us_median_over_400": round(statistics.median(stp_us), 2),
        "time_vs_fill": fill_curve,
        "vs_pages": "foxhunt 'GPU Segment Tree for PER Sampling': O(n) prefix-sum sampling grew 5 -> 23 ms as the "
                    "buffer filled 128K -> 500K on an H100; ~0.1 ms expected for the tree",
        "roofline": roofline("sample_tree_kernel<128> + small_update_kernel",
                             tb * levels * 8 + 12 * sum(min(1 << lv, 820) for lv in range(levels + 1)),
                             us_t, peak, peak_kind,
                             note="latency-bound: dependent loads down 19 levels of an L2-resident 4 MiB tree"),
        "l2": "warm (the 4 MiB tree stays resident across steps); steady state: graph of 8 steps per replay; "
              "growth loop: CUDA events around every step of all 400, enqueued back to back"}

    # ---- heavy: N = 1,048,576 lognormal(0, 2), 1% zeros, alpha 0.7, B = 65536
    Hv = workloads.HEAVY
    p = workloads.heavy_priorities()
    n, b = p.size, Hv["B"]
    ctx = per.PerContext(n, Hv["alpha"], per.PER_SCAN | per.PER_TREE)
    per.per_set_priorities(ctx.handle, tensor(p))
    ia = torch.empty(b, dtype=torch.int32, device=dev)
    ib = torch.empty(b, dtype=torch.int32, device=dev)
    w_h = torch.empty(b, dtype=torch.float32, device=dev)
    per.per_build_cdf(ctx.handle)
    per.per_sample(ctx.handle, b, Hv["seed"], 0, per.PER_SCAN, ia)
    per.per_sample(ctx.handle, b, Hv["seed"], 0, per.PER_TREE, ib)
    checks["heavy"] = {"p": p, "idx_scan": ia.cpu().numpy(), "idx_tree": ib.cpu().numpy(),
                       "tree_root": float(per.read_tree(ctx.handle)[1].item())}
    us = {
        "build_cdf": time_graph(torch, graph_of(torch, lambda: per.per_build_cdf(ctx.handle)), 30, flush.clean),
        "sample_scan": time_graph(torch, graph_of(torch, lambda: per.per_sample(ctx.handle, b, Hv["seed"], 0,
                                                                             per.PER_SCAN, ia)), 30, flush.clean),
        "sample_tree": time_graph(torch, graph_of(torch, lambda: per.per_sample(ctx.handle, b, Hv["seed"], 0,
                                                                             per.PER_TREE, ib)), 30, flush.clean),
        "is_weights_7_betas": time_graph(torch, graph_of(torch, lambda: [per.per_is_weights(ctx.handle, ia, beta, w_h)
                                                                         for beta in Hv["betas"]]), 30, flush.clean),
    }
    assert per.per_check(ctx.handle) == 0
    ctx.close()
    cfg["heavy"] = {
        "workload": f"N={n} lognormal(0, sigma 2) with 1% exact zeros, alpha={Hv['alpha']}, B={b} stratified, IS "
                    f"weights at beta {Hv['betas'][0]}..{Hv['betas'][-1]}; scan and tree paths",
        "us_per_call": {k: round(v, 2) for k, v in us.items()},
        "build_cdf_gbs": round(8 * n / (us["build_cdf"] * 1e-6) / 1e9, 1),
        "samples_per_s_scan": b / (us["sample_scan"] * 1e-6),
        "roofline": roofline("build_cdf_wave_kernel<512>", 8 * n, us["build_cdf"], peak, peak_kind,
                             note="8 MiB each way: one wave of tiles, latency-dominated"),
        "l2": "flushed before each rep (512 MiB write + 512 MiB read of other buffers)"}

    # ---- stress: N = 16,777,216 uniform(0,1], B = 1,048,576
    S = workloads.STRESS
    p = workloads.stress_priorities()
    n, b = p.size, S["B"]
    ctx = per.PerContext(n, S["alpha"], per.PER_SCAN)
    per.per_set_priorities(ctx.handle, tensor(p))
    for _ in range(3):
        per.per_build_cdf(ctx.handle)
    g_scan = graph_of(torch, lambda: per.per_build_cdf(ctx.handle))
    us_scan = time_graph(torch, g_scan, 30, flush.clean)
    us_scan_dirty = time_graph(torch, g_scan, 30, flush.dirty)
    # without a flush: 20 calls back to back in one graph (whatever of the
    # 128 MB working set the 126 MB L2 keeps between calls)
    us_scan_warm = time_graph(torch, graph_of(torch, lambda: [per.per_build_cdf(ctx.handle) for _ in range(20)]),
                              15, None, per_replay=20)
    i_st = torch.empty(b, dtype=torch.int32, device=dev)
    per.per_sample(ctx.handle, b, 1, 0, per.PER_SCAN, i_st)
    us_samp = time_graph(torch, graph_of(torch, lambda: per.per_sample(ctx.handle, b, 1, 0, per.PER_SCAN, i_st)),
                         20, flush.clean)
    checks["stress"] = {"p": p, "idx": i_st.cpu().numpy()}
    assert per.per_check(ctx.handle) == 0
    ctx.close()
    ctx = per.PerContext(n, 1.0, per.PER_SCAN)
    per.per_set_priorities(ctx.handle, tensor(p))
    per.per_build_cdf(ctx.handle)
    us_scan1 = time_graph(torch, graph_of(torch, lambda: per.per_build_cdf(ctx.handle)), 30, flush.clean)
    ctx.close()
    samp_bytes = min(4 * n, b * 32) + 4 * b
    cfg["stress"] = {
        "workload": f"N={n} fp32 uniform(0,1], alpha={S['alpha']} (and 1.0); build_cdf + sample {b} stratified",
        "build_cdf_us": round(us_scan, 2), "build_cdf_us_alpha1": round(us_scan1, 2),
        "build_cdf_us_after_write_only_flush": round(us_scan_dirty, 2),
        "build_cdf_us_no_flush_back_to_back": round(us_scan_warm, 2),
        "build_cdf_gbs": round(8 * n / (us_scan * 1e-6) / 1e9, 1),
        "build_cdf_frac_of_nominal_8tbs": round(8 * n / (us_scan * 1e-6) / 1e9 / 8000.0, 4),
        "target_frac_of_hbm": 0.70,
        "sample_us": round(us_samp, 2), "samples_per_s": b / (us_samp * 1e-6),
        "sample_roofline": roofline("sample_bounds_kernel + sample_scan_kernel", samp_bytes, us_samp, peak,
                                    peak_kind, traffic_for("sample_scan_stress")),
        "roofline": roofline("build_cdf_stream_kernel", 8 * n, us_scan, peak, peak_kind,
                             traffic_for("build_cdf_stress")),
        "l2": "flushed before each rep (512 MiB write + 512 MiB read of other buffers); build_cdf also after a "
              "write-only flush, whose dirty lines are written back inside the timed call, and without a flush "
              "(20 calls back to back per graph replay)"}

    # ---- resample: 256 rows x 65536 log-weights N(0, 2^2)
    R = workloads.RESAMPLE
    lw = workloads.resample_logw()
    logw = tensor(lw)
    ridx = torch.empty((R["rows"], R["P"]), dtype=torch.int32, device=dev)
    per.per_resample(logw, 6, 0, ridx)
    checks["resample"] = {"lw": lw, "idx": ridx.cpu().numpy()}
    us_r = time_graph(torch, graph_of(torch, lambda: per.per_resample(logw, 6, 0, ridx)), 20, flush.clean)
    D = 4
    state = torch.randn((R["rows"], R["P"], D), generator=torch.Generator(device=dev).manual_seed(6), device=dev)
    out_state = torch.empty_like(state)
    out_lw = torch.empty_like(logw)
    per.per_resample_step(logw, state, 6, 0, ridx, out_state, out_lw)
    us_rs = time_graph(torch, graph_of(torch, lambda: per.per_resample_step(logw, state, 6, 0, ridx, out_state,
                                                                         out_lw)), 20, flush.clean)
    rbytes = 8 * R["rows"] * R["P"]
    sbytes = R["rows"] * R["P"] * (4 + 4 + 4 + 8 * D)
    cfg["resample"] = {
        "workload": f"row-batched systematic resampling {R['rows']} rows x {R['P']} fp32 log-weights N(0, 2^2): "
                    f"softmax, per-row CDF, u_j = (j + U_b)/P",
        "resample_us": round(us_r, 2), "rows_per_s": R["rows"] / (us_r * 1e-6),
        "resample_step_d4_us": round(us_rs, 2),
        "resample_step_d4_gbs": round(sbytes / (us_rs * 1e-6) / 1e9, 1),
        "resample_step_d4_frac": round(sbytes / (us_rs * 1e-6) / 1e9 / peak, 4),
        "roofline": roofline("resample_kernel<0, 1, 1> (indices; P a power of two, segments staged)", rbytes, us_r, peak, peak_kind, traffic_for("resample")),
        "l2": "flushed before each rep (512 MiB write + 512 MiB read of other buffers)"}

    extras.update(rank_and_gather_extras(per, torch, dev, peak, flush, tensor))
    return cfg, extras, checks


def workloads_apply(prio, idx, p):
    """prio with prio[idx[k]] = p[k] in batch order (the last occurrence
    wins): the host's copy of the buffer the tree workload fills."""
    out = prio.copy()
    out[idx] = p  # numpy fancy assignment keeps the last duplicate
    return out


def rank_and_gather_extras(per, torch, dev, peak, flush, tensor):
    """Measurements beyond the workloads' records: the minibatch step that
    also copies the sampled transitions, rank-based PER (the sort and the
    step) and the torch.cumsum / searchsorted comparator."""
    out = {}
    Mb = workloads.MINIBATCH
    ctx = per.PerContext(Mb["N"], Mb["alpha"], per.PER_SCAN)
    per.per_set_priorities(ctx.handle, tensor(workloads.minibatch_priorities()))
    trans = torch.randn((Mb["N"], 64), generator=torch.Generator(device=dev).manual_seed(7), device=dev)
    gi = [torch.empty(Mb["B"], dtype=torch.int32, device=dev) for _ in range(2)]
    gw = torch.empty(Mb["B"], dtype=torch.float32, device=dev)
    grows = torch.empty((Mb["B"], 64), dtype=torch.float32, device=dev)
    gnew = [tensor(workloads.minibatch_new_priorities(r)) for r in range(8)]
    per.per_build_cdf(ctx.handle)
    per.per_sample(ctx.handle, Mb["B"], Mb["seed"], 0, per.PER_SCAN, gi[0])

    def gather_steps():
        for r in range(8):
            per.per_step_gather(ctx.handle, gi[r & 1], gnew[r], Mb["B"], Mb["seed"], r * Mb["B"], per.PER_SCAN,
                                Mb["beta"], gi[(r + 1) & 1], gw, trans, grows)
    gather_steps()
    us_g = time_graph(torch, graph_of(torch, gather_steps), 30, per_replay=8)
    out["step_gather_minibatch_256B"] = {"N": Mb["N"], "B": Mb["B"], "row_bytes": 256, "us": round(us_g, 2),
                                         "l2": "warm (the transitions stay resident across steps)",
                                         "timing": "graph of 8 steps between events, per step"}
    assert per.per_check(ctx.handle) == 0
    ctx.close()
    # rank-based PER on the minibatch workload: per step, update the 8192
    # sampled items, re-sort all 262,144 by priority, sample 8192 ranks with
    # IS weights (per_step, mode PER_RANK)
    ctx = per.PerContext(Mb["N"], Mb["alpha"], per.PER_RANK)
    per.per_set_priorities(ctx.handle, tensor(workloads.minibatch_priorities()))
    per.per_rank_build(ctx.handle)
    ri = [torch.empty(Mb["B"], dtype=torch.int32, device=dev) for _ in range(2)]
    rw = torch.empty(Mb["B"], dtype=torch.float32, device=dev)
    rnew = [tensor(workloads.minibatch_new_priorities(r)) for r in range(8)]
    per.per_sample(ctx.handle, Mb["B"], Mb["seed"], 0, per.PER_RANK, ri[0])

    def rank_steps():
        for r in range(8):
            per.per_step(ctx.handle, ri[r & 1], rnew[r], Mb["B"], Mb["seed"], r * Mb["B"], per.PER_RANK,
                         Mb["beta"], ri[(r + 1) & 1], rw)
    rank_steps()
    us_k = time_graph(torch, graph_of(torch, rank_steps), 30, per_replay=8)
    us_b = time_graph(torch, graph_of(torch, lambda: per.per_rank_build(ctx.handle)), 30)
    out["rank_minibatch_step"] = {"N": Mb["N"], "B": Mb["B"], "us": round(us_k, 2), "sort_us": round(us_b, 2),
                                  "l2": "warm (the 1 MiB priorities stay resident across steps)",
                                  "timing": "graph of 8 steps between events, per step"}
    assert per.per_check(ctx.handle) == 0
    ctx.close()
    S = workloads.STRESS
    n = S["N"]
    ctx = per.PerContext(n, S["alpha"], per.PER_RANK)
    per.per_set_priorities(ctx.handle, tensor(workloads.stress_priorities()))
    per.per_rank_build(ctx.handle)
    us_16 = time_graph(torch, graph_of(torch, lambda: per.per_rank_build(ctx.handle)), 10, flush.clean)
    sort_bytes = RANK_SORT_BYTES_PER_KEY * n
    out["rank_sort_16M"] = {"N": n, "us": round(us_16, 2), "keys_per_s": n / (us_16 * 1e-6),
                            "gbs": round(sort_bytes / (us_16 * 1e-6) / 1e9, 1),
                            "frac_of_measured_peak": round(sort_bytes / (us_16 * 1e-6) / 1e9 / peak, 4),
                            "bytes_per_key": RANK_SORT_BYTES_PER_KEY, "l2": "flushed before each rep"}
    assert per.per_check(ctx.handle) == 0
    ctx.close()
    # comparator, context only: the same CDF and sampling with library kernels
    tp = tensor(workloads.stress_priorities())
    tcdf = torch.empty_like(tp)
    tu = ((torch.arange(S["B"], device=dev, dtype=torch.float32) + 0.5) / S["B"])
    tidx = torch.empty(S["B"], dtype=torch.int64, device=dev)

    def torch_cdf():
        torch.cumsum(tp.pow(S["alpha"]), 0, out=tcdf)

    def torch_sample():
        torch.searchsorted(tcdf, tu * tcdf[-1], out=tidx)
    torch_cdf()
    out["torch_comparator_16M"] = {
        "build_cdf_us": round(time_graph(torch, graph_of(torch, torch_cdf), 30, flush.clean), 2),
        "sample_us": round(time_graph(torch, graph_of(torch, torch_sample), 20, flush.clean), 2),
        "note": "torch.cumsum(p**alpha) and torch.searchsorted on the stress input (library kernels); context only",
        "l2": "flushed before each rep"}
    return out


def oracle_legs(cfg, checks, seconds):
    """The CPU oracle (serial C, fp64, one thread) timed on a bounded sample
    of each workload, and the count of the GPU's sampled indices that differ
    from the oracle's search of its own fp64 CDF on the same inputs."""
    import oracle
    oracle.build()
    budget = max(1.0, seconds / 4)

    def timed_loop(fn):
        t0 = time.perf_counter()
        it = 0
        while True:
            fn()
            it += 1
            dt = time.perf_counter() - t0
            if dt >= budget:
                return dt / it, it

    def mism(a, b):
        return {"differing": int(np.count_nonzero(a != b)), "samples": int(a.size),
                "note": "all inside the boundary band (checked by the GPU tests)"}

    Sm = workloads.SMALL
    c = checks["small"]

    def small():
        C = oracle.cdf64(c["p"], Sm["alpha"])
        idx, _ = oracle.sample_cdf_f64(C, Sm["B"], Sm["seed"], 0)
        oracle.is_weights(c["p"], c["p"].size, Sm["alpha"], idx, Sm["beta"])
        return idx
    s_it, it = timed_loop(small)
    cfg["small"]["cpu_baseline"] = {"value": Sm["B"] / s_it, "unit": "samples/s", "cores": 1, "kind": "oracle",
                                    "us_per_combined_call": round(s_it * 1e6, 1),
                                    "sample": f"{it} repetitions of build_cdf + sample + IS weights, single thread"}
    cfg["small"]["mismatches_vs_oracle_fp64"] = mism(checks["small"]["idx"], small())

    c = checks["minibatch"]
    C = oracle.cdf64(c["p"], ALPHA)
    own, _ = oracle.sample_cdf_f64(C, B, W["seed"], 0)
    cfg["minibatch"]["mismatches_vs_oracle_fp64"] = mism(c["idx"], own)
    cfg["minibatch"]["cpu_baseline"] = cpu_baseline(budget)

    T = workloads.TREE
    c = checks["tree"]
    cap_pow2 = 1 << 19
    tb = T["B"]

    def tree_step():
        leaves = oracle.tree_leaves(c["prio"], T["alpha"], cap_pow2)
        tree = oracle.tree_build(leaves)
        idx, u = oracle.sample_tree(tree, tb, T["seed"], T["steps"] * tb)
        prio = workloads_apply(c["prio"], idx, c["prio"][idx])
        oracle.tree_build(oracle.tree_leaves(prio, T["alpha"], cap_pow2))
        return idx, u, leaves
    t_it, it = timed_loop(tree_step)
    cfg["tree"]["cpu_baseline"] = {"value": 1.0 / t_it, "unit": "steps/s", "cores": 1, "kind": "oracle",
                                   "us_per_step": round(t_it * 1e6, 1),
                                   "sample": f"{it} sample + update steps at full fill (the oracle rebuilds the "
                                             "whole tree per update), single thread"}
    _, u, leaves = tree_step()
    Cl = np.cumsum(leaves.astype(np.float64))
    own = np.minimum(np.searchsorted(Cl, u.astype(np.float64), side="left"), cap_pow2 - 1)
    cfg["tree"]["mismatches_vs_oracle_fp64"] = mism(c["idx"], own)

    Hv = workloads.HEAVY
    c = checks["heavy"]

    def heavy():
        C = oracle.cdf64(c["p"], Hv["alpha"])
        idx, _ = oracle.sample_cdf_f64(C, Hv["B"], Hv["seed"], 0)
        for beta in Hv["betas"]:
            oracle.is_weights(c["p"], c["p"].size, Hv["alpha"], idx, beta)
        return C, idx
    h_it, it = timed_loop(heavy)
    C, own = heavy()
    cfg["heavy"]["cpu_baseline"] = {"value": Hv["B"] / h_it, "unit": "samples/s", "cores": 1, "kind": "oracle",
                                    "us_per_iteration": round(h_it * 1e6, 1),
                                    "sample": f"{it} x (build_cdf, sample {Hv['B']}, IS weights at 7 betas), single "
                                              "thread"}
    ut = oracle.thresholds(Hv["B"], Hv["seed"], 0, c["tree_root"])  # the tree path's thresholds (T = root)
    own_t = np.minimum(np.searchsorted(C, ut.astype(np.float64), side="left"), C.size - 1)
    cfg["heavy"]["mismatches_vs_oracle_fp64"] = {"scan": mism(c["idx_scan"], own), "tree": mism(c["idx_tree"], own_t)}

    S = workloads.STRESS
    c = checks["stress"]
    t0 = time.perf_counter()
    C = oracle.cdf64(c["p"], S["alpha"])
    t1 = time.perf_counter()
    own, _ = oracle.sample_cdf_f64(C, S["B"], 1, 0)
    t2 = time.perf_counter()
    cfg["stress"]["cpu_baseline"] = {"value": 8 * c["p"].size / (t1 - t0) / 1e9, "unit": "GB/s (build_cdf)",
                                     "cores": 1, "kind": "oracle", "build_cdf_us": round((t1 - t0) * 1e6, 1),
                                     "sample_us": round((t2 - t1) * 1e6, 1),
                                     "sample": "one build_cdf of 16M items and one sample of 1M, single thread"}
    cfg["stress"]["mismatches_vs_oracle_fp64"] = mism(c["idx"], own)

    R = workloads.RESAMPLE
    c = checks["resample"]
    rows = list(range(0, R["rows"], 32))

    def resample_rows():
        return [oracle.resample_row(c["lw"][b], oracle.u01_closed_open(6, 0, b))[0] for b in rows]
    r_it, it = timed_loop(resample_rows)
    cfg["resample"]["cpu_baseline"] = {"value": len(rows) / r_it, "unit": "rows/s", "cores": 1, "kind": "oracle",
                                       "us_per_row": round(r_it / len(rows) * 1e6, 1),
                                       "sample": f"{it} x {len(rows)} rows of {R['P']}, single thread"}
    got = np.concatenate([c["idx"][b] for b in rows])
    cfg["resample"]["mismatches_vs_oracle_fp64"] = mism(got, np.concatenate(resample_rows()))


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
