"""Benchmark of the verify-and-recover step on GB300.

One step = the whole hot path on one batch of the large-batch mixed-sampling
workload (B=512, k=7, f=4, V=151936, fp32 logits, T=0 on half the rows and
U(0.5,1.2) on the rest): one SSD round through ssd_verify_fork_cache (row
statistics, acceptance, first-reject prefix, recovery/bonus draw, forked
top-f, then the speculation-cache step: clear, insert the forked recovery
tokens -- on a side stream during the draw -- and look up each row's
realised outcome).  The metric is verified batch rows per second; the
roofline object reports the achieved HBM bandwidth of the dominant unit, the
streaming statistics pass (its two kernels run concurrently on two streams and
are timed together from the fork to the join).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

N > 1 runs under torch.distributed.run, one process per GPU, each on its own
batch (weak scaling, no collective on the data path).  `--impl reference`
times the CPU oracle on a bounded sample of the same workload instead.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "mixed512"
METRIC = "verify+recover rows/s"
UNIT = "rows/s"
FALLBACK_HBM_GBS = 6800.0
CACHE_DEPTH = 7
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "stats_pass_mixed512.md")
NOMINAL_HBM_GBS = 8000.0
KERNEL_SOURCES = ["speculative_decoding_verification_70_gb300/csrc/ssd_stats.cu",
                  "speculative_decoding_verification_70_gb300/csrc/ssd_pass.cuh",
                  "speculative_decoding_verification_70_gb300/csrc/ssd_scan.cuh",
                  "speculative_decoding_verification_70_gb300/csrc/ssd_device.cuh",
                  "speculative_decoding_verification_70_gb300/csrc/ssd_layout.h"]


def kernel_source_hash():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as fh:
                d = json.load(fh)
            v = d.get("hbm_gbs")
            if isinstance(v, dict):
                v = v.get("value") or v.get("gbs")
            if v:
                return float(v), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def ncu_traffic_per_launch():
    """DRAM bytes (read + write) of one statistics pass at full size from the
    committed ncu summary, if it was taken on the current kernel sources."""
    if not os.path.exists(PROFILE_SUMMARY):
        return None
    want = kernel_source_hash()
    with open(PROFILE_SUMMARY) as fh:
        for line in fh:
            if line.startswith("machine:"):
                try:
                    d = json.loads(line[len("machine:"):])
                except ValueError:
                    return None
                if d.get("kernel_source_hash") == want:
                    return d.get("dram_bytes_per_launch_full")
    return None


class ClockSampler:
    """nvidia-smi clock and throttle sampling during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(ms, world, device=None):
    """The largest per-rank time; every rank receives it (an all-reduce MAX
    over the default process group when world > 1)."""
    if world == 1:
        return float(ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(B, world, ms_max, steps):
    """Whole-job rows per second: every rank verifies B rows per step, and the
    job takes as long as its slowest rank."""
    return world * B / (ms_max / 1e3 / steps)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
class Step:
    """Device buffers and one step of the hot path."""

    def __init__(self, ssd, w, inp, dev):
        import torch
        self.ssd, self.w, self.inp = ssd, w, inp
        self.ws = ssd.new_workspace(ssd.workspace_bytes(w.B, w.k, w.V, w.f), dev)
        self.out = {}
        self.cache = ssd.SpecCache(1 << max(1, (2 * w.B * (w.k + 1) * w.f - 1).bit_length()),
                                   CACHE_DEPTH)
        g = torch.Generator(device=dev)
        g.manual_seed(99)
        self.payload = torch.randint(0, w.V, (w.B * (w.k + 1) * w.f, CACHE_DEPTH),
                                     generator=g, device=dev, dtype=torch.int32)
        self.look = None

    def __call__(self):
        # one SSD round: verify + forks, the forks into the (cleared) cache on
        # a side stream during the recovery draw, the outcome looked up
        i = self.inp
        o = self.ssd.ssd_verify_fork_cache(i["Z"], i["D"], i["x"], i["T"], i["u_acc"],
                                           i["u_smp"], self.w.f, i["mask"], self.cache,
                                           self.payload, ws=self.ws, out=self.out)
        self.look = o
        return o


def b1_latency(ssd, W, dev, reps=300):
    """Latency of the B = 1 SSD step (ssd_fork: k=7, f=3, V=128256 bf16,
    T=1; verify + forked recovery + cache clear/insert/lookup), launched
    eagerly and replayed as a captured CUDA graph; microseconds per step."""
    import torch
    w = W.workload("ssd_fork")
    inp = W.make_inputs(w, device=dev, seed=W.default_seed("ssd_fork"))
    step = Step(ssd, w, inp, dev)
    stream = torch.cuda.current_stream()

    def timed(fn):
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps

    eager = timed(step)
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for _ in range(3):
            step()
    stream.wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    graph = timed(g.replay)
    step.cache.close()
    return {"workload": "ssd_fork: B=1 k=7 f=3 V=128256 bf16, T=1, verify+fork+cache step",
            "eager_us": round(eager, 2), "graph_us": round(graph, 2)}


def config_throughput(ssd, W, dev, name, temp=None, sets=128, rounds=10, peak=None):
    """One workload of the table in its own launch configuration, measured
    like the headline step: ms per call with CUDA events over `rounds`
    passes through `sets` input sets (the sets together are larger than L2,
    so each call streams its logits from HBM), rows/s, and GB/s over the
    algorithmic bytes (every logit row read once: the 2k+1 rows of the
    verify plus, for the SSD round step, draft row k).  B = 1 workloads are
    also captured as one CUDA graph of `sets` steps (per-step time of the
    replay).  The SSD workloads run ssd_verify_fork_cache (verify + forks +
    cache clear / insert / outcome lookup), the sync one ssd_verify."""
    import torch
    w = W.workload(name)
    forks = w.ssd and w.f > 0
    s = 4 if w.dtype == "f32" else 2
    rows_read = (2 * w.k + 1) + (1 if forks else 0)
    step_bytes = w.B * rows_read * w.V * s
    # enough sets to hold 3x the 129 MB L2 (at most `sets`, at least 2)
    nsets = max(2, min(sets, -(-3 * 129 * 2 ** 20 // step_bytes)))
    inp = W.make_inputs(W.workload(name, B=w.B * nsets), device=dev,
                        seed=W.default_seed(name) + 17, temp=temp)
    stream = torch.cuda.current_stream()
    ws = ssd.new_workspace(ssd.workspace_bytes(w.B, w.k, w.V, w.f if forks else 0), dev)
    cache = ssd.SpecCache(1 << max(6, (2 * w.B * (w.k + 1) * w.f - 1).bit_length()),
                          CACHE_DEPTH) if forks else None
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    payload = torch.randint(0, w.V, (w.B * (w.k + 1) * max(w.f, 1), CACHE_DEPTH), generator=g,
                            device=dev, dtype=torch.int32)
    views = []
    for i in range(nsets):
        sl = slice(i * w.B, (i + 1) * w.B)
        views.append(({key: v[sl] for key, v in inp.items()}, {}))

    def call(i):
        v, o = views[i]
        if forks:
            ssd.ssd_verify_fork_cache(v["Z"], v["D"], v["x"], v["T"], v["u_acc"], v["u_smp"],
                                      w.f, v["mask"], cache, payload, ws=ws, out=o)
        else:
            ssd.ssd_verify(v["Z"], v["D"], v["x"], v["T"], v["u_acc"], v["u_smp"], ws=ws, out=o)

    def sweep():
        for i in range(nsets):
            call(i)

    def timed(fn, n):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    ms = timed(sweep, rounds) / nsets
    prof_stats = prof_span = None
    if w.B > 1:   # the statistics pass as a phase (fork to join), per-launch events
        ssd.profile_begin(16 * nsets)
        sweep()
        torch.cuda.synchronize()
        prof = ssd.profile_end()
        if prof.get("stats_pass", {}).get("timed"):
            prof_stats = prof["stats_pass"]["total_ms"] / prof["stats_pass"]["timed"]
        if prof.get("stats_span", {}).get("timed"):
            prof_span = prof["stats_span"]["total_ms"] / prof["stats_span"]["timed"]
    peak = peak or measured_peaks()[0]
    vb = w.B * (2 * w.k + 1) * w.V * s + (w.B * w.V * s if forks else 0)
    res = {"workload": "%s: B=%d k=%d%s V=%d %s, T=%s" % (
               name, w.B, w.k, (" f=%d" % w.f) if forks else "", w.V, w.dtype,
               temp if temp is not None else w.temp),
           "call": "ssd_verify_fork_cache" if forks else "ssd_verify",
           "us_per_step": round(ms * 1e3, 2), "rows_per_s": round(w.B / (ms / 1e3), 1),
           "algorithmic_bytes": vb, "gbs": round(vb / (ms / 1e3) / 1e9, 1),
           "frac_of_measured_peak": round(vb / (ms / 1e3) / 1e9 / peak, 4),
           "input_sets": nsets, "l2": "each call reads a set not touched since %d calls ago"
                                     % (nsets - 1)}
    if prof_stats:
        res["stats_pass_ms"] = round(prof_stats, 5)
        res["stats_pass_gbs"] = round(vb / (prof_stats / 1e3) / 1e9, 1)
        res["stats_pass_frac_of_measured_peak"] = round(vb / (prof_stats / 1e3) / 1e9 / peak, 4)
    if prof_span:  # the two statistics kernels' own span (no fork / join)
        res["stats_kernels_ms"] = round(prof_span, 5)
        res["stats_kernels_gbs"] = round(vb / (prof_span / 1e3) / 1e9, 1)
        res["stats_kernels_frac_of_measured_peak"] = round(vb / (prof_span / 1e3) / 1e9 / peak, 4)
    if w.B == 1:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            sweep()
        stream.wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            sweep()
        res["graph_us_per_step"] = round(timed(graph.replay, rounds) / nsets * 1e3, 2)
    if cache is not None:
        cache.close()
    del inp, views
    return res


def draft_pipeline(ssd, w, inp, dev, reps=50):
    """The drafter's side fused with the verify (the next step of the hot
    path): ssd_draft_sample over the k+1 SSD draft rows (Gumbel-max tokens,
    the draft rows' statistics and the f forks with the drafted token masked)
    followed by ssd_verify_drafted, which streams only the target rows.
    Milliseconds per call, CUDA events, same workload."""
    import torch
    ws = ssd.new_workspace(ssd.workspace_bytes(w.B, w.k, w.V, w.f + 1), dev)
    dout, vout = {}, {}
    x = torch.empty((w.B, w.k), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def draft():
        ssd.ssd_draft_sample(inp["D"], inp["T"], w.k, 1234, 0, f=w.f, ws=ws, out=dout)

    def verify():
        x.copy_(dout["x"][:, : w.k])
        ssd.ssd_verify(inp["Z"], inp["D"], x, inp["T"], inp["u_acc"], inp["u_smp"],
                       drafted=True, ws=ws, out=vout)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    draft()
    t_d = timed(draft)
    t_v = timed(verify)
    row = w.B * (w.k + 1) * w.V * 4
    return {"draft_sample_ms": round(t_d, 4), "verify_drafted_ms": round(t_v, 4),
            "draft_sample_gbs": round(row / (t_d / 1e3) / 1e9, 1),
            "verify_drafted_stream_gbs": round(row / (t_v / 1e3) / 1e9, 1)}


def topk_verify(ssd, w, inp, dev, K=32, top_p=0.9, reps=50):
    """Verify over top-K / top-p filtered distributions on the same workload
    (one pass over the 2k+1 rows, no exponentials in it; the rest on at most
    K candidates per row).  Milliseconds per call and the pass's GB/s."""
    import torch
    D = inp["D"][:, : w.k].contiguous()
    tp = torch.full((w.B,), top_p, dtype=torch.float32, device=dev)
    out = {}
    ws = ssd.new_workspace(ssd.load_library().ssd_topk_workspace_bytes(w.B, w.k, w.V, K), dev)

    def call():
        ssd.ssd_verify_topk(inp["Z"], D, inp["x"], inp["T"], K, tp, inp["u_acc"], inp["u_smp"],
                            ws=ws, out=out)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    nbytes = w.B * (2 * w.k + 1) * w.V * 4
    res = {"K": K, "top_p": top_p, "ms": round(ms, 4),
           "rows_per_s": round(w.B / (ms / 1e3), 1),
           "stream_gbs": round(nbytes / (ms / 1e3) / 1e9, 1),
           "path": "per-chunk top-K lists" if min(K, w.V) <= 32 else
                   "threshold on the token order (histogram, band, exact cut)"}
    if min(K, w.V) > 32:
        ssd.profile_begin(16 * reps)
        for _ in range(reps):
            call()
        torch.cuda.synchronize()
        prof = ssd.profile_end()
        res["ms_by_kernel"] = {k: round(v["total_ms"] / max(1, v["timed"]), 4)
                               for k, v in prof.items()}
    return res


def tree_verify(ssd, W, dev, reps=20):
    """Token-tree verification on the tree workload (64 batch rows, trees of
    widths (4, 2, 1) = 21 nodes, V = 151936, bf16, T = 0.7): milliseconds per
    call, the statistics pass's GB/s over the rows it reads (the N target rows
    and the draft rows of nodes with children) and the walk's time."""
    import torch
    cfg = W.TREE_B64
    par = W.tree_parents(cfg["widths"])
    inp = W.make_tree_inputs(cfg["B"], par, cfg["V"], dtype=cfg["dtype"], temp=cfg["temp"],
                             z_std=cfg["z_std"], d_std=cfg["d_std"], peaks=cfg["peaks"],
                             peak_boost=cfg["peak_boost"], seed=4242, device=dev)
    B, N, V = inp["Z"].shape
    out = {}

    def call():
        return ssd.ssd_verify_tree(inp["Z"], inp["D"], inp["parent"], inp["tok"], inp["T"],
                                   inp["u_acc"], inp["u_smp"], ws=out.get("ws"), out=out)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    ssd.profile_begin(8 * reps)
    for _ in range(reps):
        call()
    torch.cuda.synchronize()
    prof = ssd.profile_end()
    per = {k: v["total_ms"] / max(1, v["timed"]) for k, v in prof.items()}
    # rows read: the N target rows and the draft rows of nodes with children
    inner = len(set(int(j) for j in par[1:]))
    nbytes = B * (N + inner) * V * inp["Z"].element_size()
    acc = out["accept_len"].float().mean().item()
    res = {"workload": "B=%d N=%d (widths %s) V=%d bf16 T=0.7" % (B, N, cfg["widths"], V),
           "rows_read_per_tree": N + inner,
           "ms": round(ms, 4), "rows_per_s": round(B / (ms / 1e3), 1),
           "mean_accepted": round(acc, 3)}
    if "stats" in per:
        res["stats_ms"] = round(per["stats"], 4)
        res["stats_gbs"] = round(nbytes / (per["stats"] / 1e3) / 1e9, 1)
    if "tree_walk" in per:
        res["walk_ms"] = round(per["tree_walk"], 4)
    del inp
    return res


def cpu_baseline_sample(inp, w, target_s=15.0, max_rows=None):
    """Time the oracle (as it stands, one host thread) on a bounded sample of
    the batch rows: verify_recover + forked_topf + the dict cache."""
    import numpy as np
    import oracle
    oracle.build()
    B = w.B if max_rows is None else min(w.B, max_rows)

    def run(rows):
        sel = {k: v[:rows].cpu() for k, v in inp.items()}
        t0 = time.perf_counter()
        ref = oracle.verify_recover(sel["Z"], sel["D"], sel["x"], sel["T"], sel["u_acc"],
                                    sel["u_smp"])
        fk = oracle.forked_topf(sel["D"], w.f, sel["mask"])
        c = oracle.SpecCacheOracle(CACHE_DEPTH)
        ft = fk["fork_tok"]
        bb = np.repeat(np.arange(rows), (w.k + 1) * w.f)
        pp = np.tile(np.repeat(np.arange(w.k + 1), w.f), rows)
        c.insert(bb, pp, ft.reshape(-1), np.zeros((ft.size, CACHE_DEPTH), dtype=np.int32))
        n = ref["accept_len"]
        c.lookup(np.arange(rows), n, ref["out_tok"][np.arange(rows), np.maximum(n, 0)])
        return time.perf_counter() - t0

    t1 = run(1)
    rows = int(max(1, min(B, target_s / max(t1, 1e-6))))
    dt = run(rows)
    return {"value": rows / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "first %d of %d batch rows of %s, one host thread, %.1f s"
                      % (rows, w.B, WORKLOAD, dt)}


def _oracle_worker(job):
    """One process of the all-cores CPU baseline: draw `rows` batch rows of
    the benchmark workload with its own seed and time the oracle's step on
    them (verify_recover + forked_topf + the dict cache)."""
    rows, seed = job
    import torch
    from speculative_decoding_verification_70_gb300 import workloads as W
    torch.set_num_threads(1)
    w = W.workload(WORKLOAD, B=rows)
    inp = W.make_inputs(w, device="cpu", seed=seed)
    t0 = time.perf_counter()
    run_oracle_step(inp, w, rows)
    return time.perf_counter() - t0


def cpu_baseline_all_cores(rows_per_core=48):
    """The oracle on every host core: one spawned process per core, each on
    its own bounded sample of the workload; throughput = all rows / the
    slowest process's oracle time."""
    import multiprocessing as mp
    import oracle
    oracle.build()
    n = len(os.sched_getaffinity(0))
    with mp.get_context("spawn").Pool(n) as pool:
        times = pool.map(_oracle_worker, [(rows_per_core, 9000 + i) for i in range(n)])
    return {"value": n * rows_per_core / max(times), "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": "%d processes x %d batch rows of %s each (own seeds); the slowest "
                      "took %.1f s" % (n, rows_per_core, WORKLOAD, max(times))}


def gpu_arm(args):
    import torch
    import torch.distributed as dist
    import speculative_decoding_verification_70_gb300 as ssd
    from speculative_decoding_verification_70_gb300 import build as _build
    from speculative_decoding_verification_70_gb300 import workloads as W

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        _build.build()
    if world > 1:
        dist.barrier()
    ssd.load_library()

    w = W.workload(WORKLOAD) if not args.batch else W.workload(WORKLOAD, B=args.batch)
    inp = W.make_inputs(w, device=dev, seed=W.default_seed(WORKLOAD) + rank)
    step = Step(ssd, w, inp, dev)
    stream = torch.cuda.current_stream()

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    barrier()
    clock = clocks.stop()
    ms = ev0.elapsed_time(ev1)
    # per-launch CUDA events (the library's profiler) on separate steps after
    # the timed region: events between the launches would hold back the
    # programmatic dependent launches of the draw, so they stay out of it
    prof_steps = max(1, min(args.steps, 50))
    ssd.profile_begin(16 * prof_steps)
    for _ in range(prof_steps):
        step()
    torch.cuda.synchronize()
    prof = ssd.profile_end()
    ms_max = max_over_ranks(ms, world, dev)
    ms_step = ms_max / args.steps
    value = job_throughput(w.B, world, ms_max, args.steps)

    # end to end through the public API with host buffers
    e2e = e2e_run(ssd, w, inp, step, dev, max(3, min(args.steps, 40)), world)

    # kernels launched per step (the profiled steps run the same schedule)
    launches = args.steps * sum(v["launches"] for v in prof.values()) // prof_steps
    per_kernel = {k: v["total_ms"] / max(1, v["timed"]) for k, v in prof.items()}
    # dominant unit: the streaming statistics pass, two kernels running
    # concurrently on two streams (target rows; SSD draft rows with the
    # forked top-f), timed as one phase from the fork to the join.  Its
    # algorithmic bytes are every logit row read once: 2 (k+1) V fp32 values
    # per batch row.
    row_bytes = w.B * (w.k + 1) * w.V * 4
    nbytes = 2 * row_bytes
    roof = None
    if prof.get("stats_pass", {}).get("timed"):
        per = per_kernel["stats_pass"]
        peak, kind = measured_peaks()
        achieved = nbytes / (per / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": ncu_traffic_per_launch(),
                "peak_kind": kind,
                "kernel": "statistics pass: stats_kernel (target rows 0..k) concurrent with "
                          "stats_kernel<top-f> (draft rows 0..k)",
                "bytes_per_launch": nbytes, "ms_per_launch": round(per, 5),
                "per_kernel_gbs": {k: round(row_bytes / (per_kernel[k] / 1e3) / 1e9, 1)
                                   for k in ("stats", "stats_topf") if k in per_kernel},
                "step_algorithmic_gbs": round(nbytes / (ms_step / 1e3) / 1e9, 1),
                # against the part's nominal HBM3e bandwidth as well (8 TB/s)
                "nominal_gbs": NOMINAL_HBM_GBS,
                "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                "ms_per_step_by_scope": {k: round(v, 5) for k, v in per_kernel.items()}}
        if prof.get("stats_span", {}).get("timed"):
            # the same pass without the fork and join: the two kernels' span
            span = per_kernel["stats_span"]
            roof["kernels_span_ms"] = round(span, 5)
            roof["kernels_span_frac"] = round(nbytes / (span / 1e3) / 1e9 / peak, 4)
    line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded; shapes and value recipe of the large-batch mixed "
                    "sampling workload)",
            "config": {"workload": "%s: B=%d k=%d f=%d V=%d fp32 logits, T=0 on half the rows, "
                                   "U(0.5,1.2) elsewhere; Zipf-placed peaks; cache depth %d"
                                   % (WORKLOAD, w.B, w.k, w.f, w.V, CACHE_DEPTH),
                       "global_batch": w.B * world, "per_gpu_batch": w.B,
                       "l2": "inputs (%.2f GB per step) larger than L2" % (nbytes / 1e9),
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "gpu_launches": launches, "roofline": roof, "clocks": clock, "e2e": e2e,
            # logit rows verified per second: the 2k+1 rows of acceptance and
            # recovery per batch row
            "logit_rows_per_s": round(value * (2 * w.k + 1), 1),
            "us_per_step": round(ms_step * 1e3, 2)}
    if rank == 0 and world == 1:
        peak = measured_peaks()[0]
        line["configs"] = {
            "llama_sd_T0": config_throughput(ssd, W, dev, "llama_sd", "0", peak=peak),
            "llama_sd_T1": config_throughput(ssd, W, dev, "llama_sd", "1.0", peak=peak),
            "ssd_fork_T0": config_throughput(ssd, W, dev, "ssd_fork", "0", peak=peak),
            "ssd_fork_T1": config_throughput(ssd, W, dev, "ssd_fork", "1.0", peak=peak),
            "qwen_b64": config_throughput(ssd, W, dev, "qwen_b64", peak=peak),
        }
        line["latency_b1"] = b1_latency(ssd, W, dev)
        line["draft_pipeline"] = draft_pipeline(ssd, w, inp, dev)
        line["topk_verify"] = topk_verify(ssd, w, inp, dev)
        line["topk_verify_k50_p09"] = topk_verify(ssd, w, inp, dev, K=50, top_p=0.9)
        line["topp_verify_full_vocab_p09"] = topk_verify(ssd, w, inp, dev, K=w.V, top_p=0.9)
        line["tree_verify"] = tree_verify(ssd, W, dev)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_sample(inp, w)
        line["cpu_baseline_all_cores"] = cpu_baseline_all_cores()
    if rank == 0:
        print(json.dumps(line), flush=True)
    step.cache.close()
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def e2e_run(ssd, w, inp, step, dev, steps, world):
    """Same metric through the public API with pinned host buffers: every step
    copies that step's inputs host->device, runs the step and reads the results
    back device->host."""
    import torch
    names = ["Z", "D", "x", "T", "u_acc", "u_smp", "mask"]
    host = {k: torch.empty(inp[k].shape, dtype=inp[k].dtype, pin_memory=True) for k in names}
    for k in names:
        host[k].copy_(inp[k])
    outs = ["accept_len", "out_tok", "fork_tok"]
    host_out = {}
    h2d = sum(host[k].numel() * host[k].element_size() for k in names)
    stream = torch.cuda.current_stream()

    def one():
        for k in names:
            inp[k].copy_(host[k], non_blocking=True)
        o = step()
        for k in outs:
            if k not in host_out:
                host_out[k] = torch.empty(o[k].shape, dtype=o[k].dtype, pin_memory=True)
            host_out[k].copy_(o[k], non_blocking=True)
        if "hit" not in host_out:
            host_out["hit"] = torch.empty(step.look["hit"].shape, dtype=torch.int32, pin_memory=True)
            host_out["tok_out"] = torch.empty(step.look["tok_out"].shape, dtype=torch.int32,
                                              pin_memory=True)
        host_out["hit"].copy_(step.look["hit"], non_blocking=True)
        host_out["tok_out"].copy_(step.look["tok_out"], non_blocking=True)

    one()
    torch.cuda.synchronize()
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    return {"value": round(world * w.B / (ms / 1e3 / steps), 1), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps}


# ---------------------------------------------------------------------------
# the reference arm: the CPU oracle
# ---------------------------------------------------------------------------
def reference_arm(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    import oracle
    from speculative_decoding_verification_70_gb300 import workloads as W
    oracle.build()
    w0 = W.workload(WORKLOAD)
    # bounded sample: rows per step chosen so that warm-up + timed steps take
    # about a minute of host time
    probe = W.make_inputs(W.workload(WORKLOAD, B=1), device="cpu", seed=W.default_seed(WORKLOAD))
    t0 = time.perf_counter()
    run_oracle_step(probe, w0, 1)
    t_row = time.perf_counter() - t0
    total = args.steps + max(3, args.warmup)
    rows = int(max(1, min(64, 60.0 / (total * max(t_row, 1e-6)))))
    w = W.workload(WORKLOAD, B=rows)
    inp = W.make_inputs(w, device="cpu", seed=W.default_seed(WORKLOAD))
    for _ in range(max(3, args.warmup)):
        run_oracle_step(inp, w, rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run_oracle_step(inp, w, rows)
    dt = time.perf_counter() - t0
    value = rows * args.steps / dt
    sample = ("%d of %d batch rows of %s per step, one host thread" % (rows, w0.B, WORKLOAD))
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; bounded sample of the workload)",
            "config": {"workload": "%s: B=%d k=%d f=%d V=%d fp32 logits (sample of %d rows per step)"
                                   % (WORKLOAD, w0.B, w0.k, w0.f, w0.V, rows)},
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    del np
    print(json.dumps(line), flush=True)


def run_oracle_step(inp, w, rows):
    import numpy as np
    import oracle
    ref = oracle.verify_recover(inp["Z"], inp["D"], inp["x"], inp["T"], inp["u_acc"], inp["u_smp"])
    fk = oracle.forked_topf(inp["D"], w.f, inp["mask"])
    c = oracle.SpecCacheOracle(CACHE_DEPTH)
    ft = fk["fork_tok"]
    bb = np.repeat(np.arange(rows), (w.k + 1) * w.f)
    pp = np.tile(np.repeat(np.arange(w.k + 1), w.f), rows)
    c.insert(bb, pp, ft.reshape(-1), np.zeros((ft.size, CACHE_DEPTH), dtype=np.int32))
    n = ref["accept_len"]
    c.lookup(np.arange(rows), n, ref["out_tok"][np.arange(rows), np.maximum(n, 0)])


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=0,
                    help="override B (profiling captures only; not the metric's workload)")
    ap.add_argument("--only", choices=["tree", "topk", "draft", "b1", "qwen_b64", "llama_sd",
                                       "ssd_fork"], default=None,
                    help="one of the next rows' measurements alone (profiling captures; "
                         "B from --batch, timed calls from --steps)")
    ap.add_argument("--topk-k", type=int, default=32, help="K of --only topk")
    ap.add_argument("--top-p", type=float, default=0.9, help="top_p of --only topk")
    args = ap.parse_args()
    if args.impl == "reference":
        reference_arm(args)
    elif args.only:
        only_arm(args)
    else:
        gpu_arm(args)


def only_arm(args):
    """One of the next rows' measurements alone, for profiler captures:
    tree (the tree workload), topk or draft (the benchmark workload), b1 (the
    B = 1 SSD step, eager then as a graph); --batch overrides B, --steps sets
    the timed calls."""
    import torch
    import speculative_decoding_verification_70_gb300 as ssd
    from speculative_decoding_verification_70_gb300 import workloads as W
    torch.cuda.set_device(0)
    reps = max(1, args.steps)
    if args.only == "tree":
        if args.batch:
            W.TREE_B64 = dict(W.TREE_B64, B=args.batch)
        res = tree_verify(ssd, W, "cuda", reps=reps)
    elif args.only == "b1":
        res = b1_latency(ssd, W, "cuda", reps=reps)
    elif args.only in ("qwen_b64", "llama_sd", "ssd_fork"):
        res = config_throughput(ssd, W, "cuda", args.only, rounds=reps)
    else:
        w = W.workload(WORKLOAD, **({"B": args.batch} if args.batch else {}))
        inp = W.make_inputs(w, device="cuda", seed=W.default_seed(WORKLOAD))
        if args.only == "topk":
            res = topk_verify(ssd, w, inp, "cuda", K=args.topk_k, top_p=args.top_p, reps=reps)
        else:
            res = draft_pipeline(ssd, w, inp, "cuda", reps=reps)
    print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
