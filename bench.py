"""Benchmark of the GB300 token sampler.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload top_p|tiny|decode|speculative|large] [--all]

A step is one ls_sample call -- the whole sampling path: route choice,
row/request mapping, one HBM pass over the logits, temperature, exact top-k /
top-p cuts, Philox Gumbel-max -- over one batch of the workload, inputs already
resident in HBM.  The default workload is the top-p-only sampler at 256 rows x
vocab 128256 bf16 (the configuration the sampler's headline metric is quoted
on).  Rows are independent, so under torchrun every rank samples its own batch
(weak scaling, no collective on the data path); the timing is the max over
ranks and `value` counts the rows of all ranks.

Timing: W warm-up steps, then exactly K steps between a barrier and
torch.cuda.synchronize(), CUDA events on the launching stream.  The K steps are
captured once into a CUDA graph (one kernel node per step) and replayed, so
the device runs them back to back rather than waiting on Python.  L2: the step
cycles through enough copies of the logits to exceed twice the 129 MB L2, so
no step finds its inputs in L2.

`--impl reference` times the CPU oracle on the same workload instead (a
deliberately slow, plain implementation on the host cores; each step is a
bounded sample of rows), under the same metric.
"""
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

import numpy as np  # noqa: E402

METRIC = "sampled rows/s and logits HBM GB/s (% of GB300 peak) at vocab 128k–262k"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0

DESCRIPTIONS = {
    "tiny": "tiny: 4 x 1000 fp32 ~N(0,2), T=1, top_k=50, top_p=0.9 (joint route)",
    "decode": "decode batch: 64 x 32000 bf16 ~N(0,3) + 5 spikes/row, mixed per-request T/top_k/top_p (joint route)",
    "top_p": "top-p only: 256 x 128256 bf16 ~N(0,3) + Zipf(1.1) head over 200 ids, T=0.8, top_p=0.9 (top-p route)",
    "speculative": "speculative verify: 128 decode x (1+4) + 32 prefill = 672 rows gathered from 1024 x 151936 bf16 "
                   "~N(0,3), top_k in {20,40}, top_p=0.95 (joint route)",
    "large": "large: 1024 x 262144 fp32 ~N(0,4) + Zipf head, per-request mix of no filter / top_k / top_p / joint, "
             "T ~ U[0.3,1.5] (joint route)",
}


def source_hash():
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "logits_sampling_gb300", "csrc")
    for name in sorted(os.listdir(pkg)):
        if name.endswith((".cu", ".cuh")):
            h.update(open(os.path.join(pkg, name), "rb").read())
    h.update(open(os.path.join(ROOT, "include", "ls_sampler.h"), "rb").read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return json.load(open(path)), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def traffic_key(workload, call, route, split=0):
    """Key of profiles/traffic.json: the call on the workload's own route and
    kernel choice, or on a forced one."""
    return f"{workload}:{call}" + ("" if route == "auto" else f":{route}") + ("" if split == 0 else f":split{split}")


def ncu_traffic(key):
    """DRAM bytes per launch of the call's dominant kernel from the committed
    ncu record (profiles/traffic.json), if it was taken on the current kernel
    sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path))
    except (OSError, ValueError):
        return None
    ent = rec.get(key)
    if not ent or ent.get("source_hash") != source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.count(",") >= 6]
        os.unlink(self.file.name)
        sm = [float(r[0]) for r in rows if r[0].strip().replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[3 + i] and "Not" not in r[3 + i]})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dist_setup(gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("LS_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


ROUTES = {"auto": None, "kp": (False, False), "k": (False, True), "p": (True, False), "none": (True, True)}


def make_workload(name, rank, route="auto", rows=0):
    """The named workload (with `rows` > 0, that many rows of it: smaller
    cases for profiler captures); `route` other than auto sets the batch flags
    (no_top_k, no_top_p) that pick the kernel's route."""
    from logits_sampling_gb300 import workloads as W
    w = W.MAKERS[name](rows=rows) if rows > 0 and name != "speculative" else W.MAKERS[name]()
    if ROUTES[route] is not None:
        w.no_top_k, w.no_top_p = ROUTES[route]
    return w


def to_device(w, device):
    import torch
    from logits_sampling_gb300 import workloads as W
    if w.dtype == W.BF16:
        return torch.from_numpy(w.logits.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(w.logits).to(device)


def cpu_oracle_rate(w, target_s=8.0, max_rows=None, threads=None):
    """Time the CPU oracle on a bounded sample of the workload's rows (on all
    the host cores this process may use, or on `threads` of them); returns
    (rows/s, seconds, rows, threads)."""
    import oracle
    from logits_sampling_gb300 import workloads as W
    threads = oracle.default_threads() if threads is None else threads
    odt = oracle.DTYPE_BF16 if w.dtype == W.BF16 else oracle.DTYPE_F32
    mapping = oracle.speculative_mapping(*w.spec) if w.spec is not None else w.token_to_request_index
    rows = w.n if max_rows is None else min(w.n, max_rows)
    g = w.gather_indices[:rows] if w.gather_indices is not None else None
    t2r = mapping[:rows] if mapping is not None else None
    done, t0 = 0, time.perf_counter()
    while True:
        oracle.sample(w.logits, odt, rows, w.temperature, w.top_k, w.top_p, w.seed, step=w.step,
                      no_top_k=w.no_top_k, no_top_p=w.no_top_p, gather_indices=g, token_to_request_index=t2r,
                      want_kept=False, nthreads=threads)
        done += rows
        el = time.perf_counter() - t0
        if el >= target_s:
            break
    return done / el, el, done, threads


def run_reference(args, world, rank):
    if rank != 0:
        return
    from logits_sampling_gb300 import workloads as W
    w = make_workload(args.workload, rank, args.route, args.rows)
    rows = min(w.n, args.ref_rows)
    # size each step so that the whole run stays within about two minutes
    t = time.perf_counter()
    cpu_oracle_rate(w, target_s=0.0, max_rows=rows)
    per_row = (time.perf_counter() - t) / rows
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows = int(max(1, min(rows, budget / max(per_row, 1e-9))))
    for _ in range(args.warmup):
        cpu_oracle_rate(w, target_s=0.0, max_rows=rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cpu_oracle_rate(w, target_s=0.0, max_rows=rows)
    el = time.perf_counter() - t0
    import oracle
    value = rows * args.steps / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": DESCRIPTIONS[args.workload], "rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": oracle.default_threads(), "kind": "oracle",
                         "sample": f"{rows} of the workload's {w.n} rows per step"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    import torch
    import logits_sampling_gb300 as ls
    from logits_sampling_gb300 import workloads as W

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    ls.load_library()
    ls.set_split_policy(args.split)
    w = make_workload(args.workload, rank, args.route, args.rows)
    x = to_device(w, device)
    copies = max(2, int(np.ceil(2.0 * L2_BYTES / max(1, x.numel() * x.element_size()))) + 1)
    copies = min(copies, args.max_copies)
    xs = [x] + [x.clone() for _ in range(copies - 1)]
    prm = ls.SamplingParams.from_host(w.temperature, w.top_k, w.top_p, w.seed, device=device)
    gather = None if w.gather_indices is None else torch.from_numpy(w.gather_indices).to(device)
    t2r = None if w.token_to_request_index is None else torch.from_numpy(w.token_to_request_index).to(device)
    out = torch.empty(w.n, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    if args.call != "sample":
        # ids plus log-prob rows plus the selected token's log-prob: one fused call,
        # or ls_sample followed by ls_log_probs (two reads of the logits)
        out_lp = torch.empty((w.n, w.vocab), dtype=torch.float32, device=device)
        out_sel = torch.empty(w.n, dtype=torch.float32, device=device)
        if w.spec is not None and t2r is None:
            D, P, S = w.spec
            r = np.arange(w.n)
            t2r = torch.from_numpy(np.where(r < D * (1 + S), r // (1 + S), D + r - D * (1 + S)).astype(np.int32))
            t2r = t2r.to(device)

    if args.call == "verify":
        # the decode requests' verify rows: sample them, then verify random drafts
        if w.spec is None:
            raise SystemExit("--call verify needs the speculative workload")
        VD, _, VS = w.spec
        vn = VD * (1 + VS)
        vgather = gather[:vn] if gather is not None else None
        cand = torch.from_numpy(np.random.default_rng(0).integers(0, w.vocab, (VD, 1 + VS)).astype(np.int32))
        cand = cand.to(device)
        vtarget = torch.empty(vn, dtype=torch.int32, device=device)
        vpred = torch.empty(vn, dtype=torch.int32, device=device)
        vai = torch.empty(vn, dtype=torch.int32, device=device)
        van = torch.empty(VD, dtype=torch.int32, device=device)
        vprm = prm.as_struct()
        vlib = ls.load_library()
        import ctypes
        from logits_sampling_gb300._binding import _dptr, _logits_desc, _stream

    def step(i, logits):
        if args.call == "verify":
            ptr, dt, rows_, V_, stride_ = _logits_desc(logits)
            st = vlib.ls_sample_verify(ptr, dt, rows_, V_, stride_, VD, 1 + VS, _dptr(vgather), ctypes.byref(vprm), i,
                                       int(w.no_top_k), int(w.no_top_p), _dptr(cand), _dptr(vtarget), _dptr(vpred),
                                       _dptr(vai), _dptr(van), None, _stream(None))
            assert st == 0, st
        elif args.call == "argmax":
            ls.argmax(logits, n=w.n, gather_indices=gather, out=out)
        elif args.call == "fused":
            ls.sample_log_probs(logits, w.n, prm, i, w.no_top_k, w.no_top_p, gather_indices=gather,
                                token_to_request_index=t2r, out=out, out_log_probs=out_lp, out_selected=out_sel)
        elif args.call == "separate":
            ls.sample(logits, w.n, prm, i, w.no_top_k, w.no_top_p, gather_indices=gather,
                      token_to_request_index=t2r, out=out)
            ls.log_probs(logits, prm, num_rows=w.n, gather_indices=gather, token_to_request_index=t2r, out=out_lp)
        elif w.spec is not None:
            D, P, S = w.spec
            ls.sample_speculative(logits, D, P, S, prm, i, w.no_top_k, w.no_top_p, gather_indices=gather, out=out)
        else:
            ls.sample(logits, w.n, prm, i, w.no_top_k, w.no_top_p, gather_indices=gather,
                      token_to_request_index=t2r, out=out)

    for i in range(args.warmup):
        step(i, xs[i % copies])
    torch.cuda.synchronize()

    def capture(n_steps, first):
        """One CUDA graph holding n_steps sampler launches (one kernel node per
        step, each with its own Philox step), so the GPU runs them back to back
        without waiting on the host."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for j in range(n_steps):
                step(first + j, xs[j % copies])
        return g

    timed_graph = capture(args.steps, args.warmup)
    soak_graph = capture(min(args.steps, 256), 0)
    torch.cuda.synchronize()

    # clocks: sample over a ~1 s soak of the same launches that runs straight into the timed region
    clk = ClockSampler(local)
    clk.start()
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak_s:
        soak_graph.replay()
        torch.cuda.synchronize()

    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    timed_graph.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = clk.stop()
    total_ms = max_over_ranks(t0.elapsed_time(t1), world, device)
    # back-to-back graph launches: the mean launch duration is the region over K
    # (it includes the few-hundred-ns gaps between kernel nodes)
    kernel_ms = total_ms / args.steps
    ms_per_step = total_ms / args.steps
    rows_per_s = world * w.n * args.steps / (total_ms * 1e-3)
    del timed_graph, soak_graph

    # end to end through the public API: pinned host inputs -> device, sample, ids -> host
    host_x = torch.from_numpy(w.logits.view(np.int16) if w.dtype == W.BF16 else w.logits).pin_memory()
    host_prm = [torch.from_numpy(a).pin_memory() for a in
                (w.temperature, w.top_k, w.top_p, w.seed.view(np.int64))]
    dev_prm = [prm.temperature, prm.top_k, prm.top_p, prm.seed]
    host_ids = torch.empty(w.n, dtype=torch.int32).pin_memory()
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    h2d = host_x.numel() * host_x.element_size() + sum(t.numel() * t.element_size() for t in host_prm)
    d2h = w.n * 4
    dx = x.view(torch.int16) if w.dtype == W.BF16 else x
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(e2e_steps):
        dx.copy_(host_x, non_blocking=True)
        for d, h in zip(dev_prm, host_prm):
            d.copy_(h, non_blocking=True)
        step(i, x)
        host_ids.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, device) / e2e_steps
    e2e_rows = world * w.n / (e2e_ms * 1e-3)

    peaks, peak_src = measured_peaks()
    alg_bytes = W.algorithmic_bytes(w)
    if args.call == "verify":  # the decode verify rows read once; ids, drafts, predicts, accept outputs
        VD, _, VS = w.spec
        vn = VD * (1 + VS)
        alg_bytes = vn * w.vocab * w.elem_bytes + vn * (28 + 4 + 4 + 4 + 4) + VD * 4
    elif args.call == "argmax":  # the rows read once, an id written per row (no parameters)
        alg_bytes = w.n * w.vocab * w.elem_bytes + w.n * (4 + (4 if w.gather_indices is not None else 0))
    elif args.call == "fused":  # one read, the log-prob rows written, id + selected log-prob per row
        alg_bytes = W.algorithmic_bytes(w, with_log_probs=True) + w.n * (28 + 8)
    elif args.call == "separate":  # the same outputs from two calls: the logits read twice
        alg_bytes = W.algorithmic_bytes(w) + W.algorithmic_bytes(w, with_log_probs=True)
    achieved = alg_bytes / (kernel_ms * 1e-3) / 1e9
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    traffic = ncu_traffic(traffic_key(args.workload, args.call, args.route, args.split))
    # kernels launched per step: the log-prob calls add the tiled write kernel
    # for batches of at most 3/4 of the SM count of rows, of at least 16384
    # entries, whose logits fit in 60% of L2 (the library's rule)
    per_step = {"sample": 1, "argmax": 1, "verify": 2}.get(args.call)
    if per_step is None:
        props = torch.cuda.get_device_properties(device)
        deferred = (w.n * 4 <= props.multi_processor_count * 3 and w.vocab >= 16384
                    and w.n * w.vocab * x.element_size() * 5 <= props.L2_cache_size * 3)
        per_step = (1 if args.call == "fused" else 2) + (1 if deferred else 0)
    line = {
        "metric": METRIC, "value": rows_per_s, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == W.BF16 else "f32", "data": "synthetic",
        "config": {"workload": DESCRIPTIONS[args.workload] + (f" [{w.n} rows]" if args.rows else ""), "rows": w.n,
                   "vocab": w.vocab, "call": args.call,
                   "split": args.split, "route": args.route,
                   "l2": f"{copies} rotating input copies ({copies * x.numel() * x.element_size() / 1e6:.0f} MB) "
                         f"> 2x L2", "parallelism": f"replicas x{world} (rows independent, no collective)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "peak_source": f"{peak_src} hbm_gbs",
                     "kernel_us": kernel_ms * 1e3, "algorithmic_bytes_per_launch": alg_bytes},
        "e2e": {"value": e2e_rows, "unit": "rows/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms},
        "gpu_launches": args.steps * per_step,
        "clocks": clocks,
        "source_hash": source_hash(),
    }
    if rank == 0 and not args.no_cpu and args.call == "sample":
        rate, el, done, threads = cpu_oracle_rate(w, target_s=args.cpu_s, max_rows=args.ref_rows)
        line["cpu_baseline"] = {"value": rate, "unit": "rows/s", "cores": threads, "kind": "oracle",
                                "sample": f"{done} rows ({min(w.n, args.ref_rows)} of the workload's {w.n} per "
                                          f"pass) in {el:.1f} s"}
        # the same oracle on one core, on a smaller sample
        rows1 = min(w.n, 8)
        rate1, el1, done1, _ = cpu_oracle_rate(w, target_s=min(3.0, args.cpu_s), max_rows=rows1, threads=1)
        line["cpu_baseline"]["single_core"] = {"value": rate1, "unit": "rows/s", "cores": 1,
                                               "sample": f"{done1} rows ({rows1} per pass) in {el1:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(DESCRIPTIONS), default="top_p")
    ap.add_argument("--all", action="store_true", help="one line per workload")
    ap.add_argument("--soak-s", type=float, default=1.0)
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-s", type=float, default=10.0)
    ap.add_argument("--ref-rows", type=int, default=64)
    ap.add_argument("--max-copies", type=int, default=8)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--rows", type=int, default=0,
                    help="rows of the workload (0: its own; speculative keeps its own) -- smaller cases for "
                         "profiler captures, not bench lines")
    ap.add_argument("--route", choices=sorted(ROUTES), default="auto",
                    help="batch flags: auto = the workload's own; kp, k, p, none = top-k and top-p, top-k only, "
                         "top-p only, no filter (the flags switch the other filters off for every row)")
    ap.add_argument("--split", type=int, default=0, choices=[0, -1, 1, 2, 4, 8],
                    help="sampling kernel: 0 = chosen from the batch shape (default); 1, 2, 4, 8 = the streaming "
                         "sampler with that many CTAs per row; -1 = the one-CTA row kernel")
    ap.add_argument("--call", choices=["sample", "fused", "separate", "argmax", "verify"], default="sample",
                    help="sample: ids (ls_sample); fused: ids, log-prob rows and selected log-probs from one "
                         "ls_sample_log_probs call; separate: ls_sample then ls_log_probs; argmax: the "
                         "all-greedy fast path (ls_argmax) on the workload's rows; verify: ls_sample_verify on "
                         "the speculative workload's decode rows")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup(args.gpus)
    names = sorted(DESCRIPTIONS) if args.all else [args.workload]
    for name in names:
        args.workload = name
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
