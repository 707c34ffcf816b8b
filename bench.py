"""Benchmark: the seven credit-assignment estimators at num_envs=4096, seq_len=128.

One step = one pass of the whole hot path over one synthetic batch: GAE,
TD(lambda) returns, discounted returns, V-trace (vs + pg advantages),
Retrace(lambda), eligibility traces and the episodic prefix sum, each on its
own inputs (so no kernel reads another's data out of L2). value = env-steps
per second with all seven outputs produced for every (env, t).

Timing: exactly --warmup untimed steps, then exactly --steps timed steps,
replayed from CUDA graphs of whole steps over 8 rotating sets of
input/output buffers whose footprint is several times the L2; CUDA events on
the launching stream, barrier + synchronize on both sides, max over ranks.
A device-side delay queued before the start event lets the host enqueue the
replays ahead, so host launch gaps do not enter the timed region.

stdout gets ONE compact JSON line (the headline: value, roofline of the
dominant kernel against the measured HBM copy bandwidth, the float64 CPU
oracle as a baseline, an end-to-end figure through pinned host buffers, SM
clocks sampled during the timed region). Everything else goes to the JSON
file named by --detail: every estimator alone, the step in several schedules
(seven streams, one stream, one rlcs_run_group call, 2 or 3 groups on their
own streams), GAE at 64 x 512, the five truncated estimators at 4096 x 128,
the long-row sweep (256 x {1024, 4096, 16384}, 8 x 131072), the extra
entry points (fused GAE + returns, affine scan, compact GAE, time-major) and
the time-major entry points at 256 x 4096, 8 x 131072 and 1024 x 4096.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--detail PATH] [--no-long-t]

Under torchrun each rank processes its own batch (rows are independent: weak
scaling, no collective on the data path).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from synthetic_rollouts import WORKLOADS, rollout  # noqa: E402

WORKLOAD = "all7_4096x128"
METRIC = "env-steps/s and achieved HBM GB/s (% of 8 TB/s) at N=4096,T=128, 1×GB300"
UNIT = "env-steps/s"
ROTATING_SETS = 8
NOMINAL_HBM_GBS = 8000.0

# Per-estimator inputs (in launch order), outputs, and algorithmic bytes per
# env-step (each input read once, each output written once; bootstrap [N]
# counted separately).
ESTIMATORS = {
    "gae": (("rewards", "values", "terminateds"), ("out",)),
    "lambda_returns": (("rewards", "values", "terminateds"), ("out",)),
    "discounted_returns": (("rewards", "terminateds"), ("out",)),
    "vtrace": (("rewards", "values", "log_rhos", "terminateds"), ("vs", "pg")),
    "retrace": (("rewards", "values", "q_values", "log_rhos", "terminateds"), ("out",)),
    "eligibility_traces": (("x", "terminateds"), ("out",)),
    "episodic_prefix_sum": (("x_int", "terminateds"), ("out",)),
}
BACKWARD = ("gae", "lambda_returns", "discounted_returns", "vtrace", "retrace")

# The five backward estimators with truncation inputs (a truncated step
# bootstraps from next_values[t]): the same calls, 8 more bytes per step.
TRUNC_IN = ("truncateds", "next_values")
TRUNCATED = {est + "_trunc": (ESTIMATORS[est][0] + TRUNC_IN, ESTIMATORS[est][1])
             for est in BACKWARD}

# Entry points beyond the seven (timed alone, reported under "next_rows").
EXTRA = {
    "gae_and_returns": (("rewards", "values", "terminateds"), ("out", "out2")),
    "affine_scan": (("a", "b", "reset"), ("out",)),
    "gae_compact": (("rewards_bf16", "values_bf16", "terminateds_u8"), ("out",)),
}
# The seven on time-major [T, N] arrays (the _tm entry points), same bytes.
EXTRA.update({est + "_tm": spec for est, spec in ESTIMATORS.items()})
ELEM_BYTES = {"rewards_bf16": 2, "values_bf16": 2, "terminateds_u8": 1}   # others: 4
SPECS = dict(ESTIMATORS, **TRUNCATED, **EXTRA)
ROW_VALUE = BACKWARD + tuple(e + "_trunc" for e in BACKWARD) + tuple(
    e + "_tm" for e in BACKWARD) + ("gae_and_returns", "affine_scan", "gae_compact")


def base_name(est):
    """The entry point's estimator: gae_trunc -> gae, vtrace_tm -> vtrace."""
    for suffix in ("_trunc", "_tm"):
        if est.endswith(suffix):
            return est[:-len(suffix)]
    return est


def kernel_source_hash():
    """Short hash of the CUDA sources, to tell whether stored ncu counters
    still describe the kernels being timed."""
    import glob
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "linear_recurrence_scan_affine_gb300", "csrc")
    for f in sorted(glob.glob(os.path.join(csrc, "*.cu*"))):
        if os.path.basename(f) == "diag.cu":  # the diagnostic, not an estimator kernel
            continue
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def bytes_per_env_step(est):
    ins, outs = SPECS[est]
    return sum(ELEM_BYTES.get(k, 4) for k in ins) + 4 * len(outs)


def bytes_per_launch(est, N, T):
    return bytes_per_env_step(est) * N * T + (4 * N if est in ROW_VALUE else 0)


# ---------------------------------------------------------------------------
# distributed plumbing (torchrun)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(dist, value, device=None):
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "clocks.mem,temperature.gpu")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, mem, temp, reasons = [], [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
            for dst, val in ((mem, parts[8:9]), (temp, parts[9:10])):
                try:
                    dst.append(float(val[0]))
                except (IndexError, ValueError):
                    pass
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "sm_min_mhz": min(sm) if sm else None,
                "mem_mhz": statistics.median(mem) if mem else None,
                "temp_c_max": max(temp) if temp else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------
def oracle_pass(oracle, src, rows, prm):
    """All seven estimators over rows [r0, r1) of the batch (float64 oracle)."""
    r0, r1 = rows
    s = {k: (v[r0:r1] if v.ndim == 2 else v[r0:r1]) for k, v in src.items()}
    g, lm = prm["gamma"], prm["lambda_"]
    B = s["bootstrap_value"]
    oracle.gae(s["rewards"], s["values"], s["terminateds"], g, lm, B)
    oracle.lambda_returns(s["rewards"], s["values"], s["terminateds"], g, lm, B)
    oracle.discounted_returns(s["rewards"], s["terminateds"], g, B)
    oracle.vtrace(s["rewards"], s["values"], s["log_rhos"], s["terminateds"], g, lm,
                  prm["rho_bar"], prm["c_bar"], B)
    oracle.retrace(s["rewards"], s["values"], s["q_values"], s["log_rhos"], s["terminateds"],
                   g, lm, prm["c_bar"], B)
    oracle.eligibility_traces(s["x"], s["terminateds"], g, lm)
    oracle.episodic_prefix_sum(s["x_int"], s["terminateds"])


def oracle_step(oracle, src, nrows, prm, pool, threads):
    """One oracle step over the first nrows rows, rows split across threads."""
    bounds = np.linspace(0, nrows, threads + 1).astype(int)
    jobs = [(int(a), int(b)) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
    list(pool.map(lambda rg: oracle_pass(oracle, src, rg, prm), jobs))


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle(src, prm, budget_s=10.0):
    """The oracle as it stands, on all host cores for about budget_s seconds,
    then on one thread for about a third of that (the single-thread figure
    rides along under "single_thread")."""
    import concurrent.futures as cf
    import oracle
    threads = cpu_threads()
    N = src["rewards"].shape[0]
    T = src["rewards"].shape[1]

    def timed(pool, nthreads, budget):
        reps, t0 = 0, time.perf_counter()
        while True:
            oracle_step(oracle, src, N, prm, pool, nthreads)
            reps += 1
            el = time.perf_counter() - t0
            if el >= budget or reps >= 10000:
                return reps, el

    with cf.ThreadPoolExecutor(threads) as pool:
        oracle_step(oracle, src, N, prm, pool, threads)  # warm (loads the library)
        reps, el = timed(pool, threads, budget_s)
    with cf.ThreadPoolExecutor(1) as pool:
        reps1, el1 = timed(pool, 1, budget_s / 3)
    return {"value": reps * N * T / el, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": "%d full %dx%d batches, all seven estimators, float64 C oracle, rows "
                      "split over %d threads, %.1f s" % (reps, N, T, threads, el),
            "single_thread": {"value": reps1 * N * T / el1, "unit": UNIT, "cores": 1,
                              "sample": "%d full batches on one thread, %.1f s" % (reps1, el1)}}


# ---------------------------------------------------------------------------
# reference arm: the oracle, timed per step
# ---------------------------------------------------------------------------
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import concurrent.futures as cf
    import oracle
    w = WORKLOADS[WORKLOAD]
    prm = dict(gamma=w.gamma, lambda_=w.lambda_, rho_bar=w.rho_bar, c_bar=w.c_bar)
    src = rollout(w.N, w.T, w.seed, w.p_term)
    threads = cpu_threads()
    with cf.ThreadPoolExecutor(threads) as pool:
        t0 = time.perf_counter()
        oracle_step(oracle, src, w.N, prm, pool, threads)
        full = time.perf_counter() - t0
        budget = 150.0  # seconds for warmup + steps
        nrows = w.N
        if full * (args.steps + args.warmup) > budget:
            nrows = max(threads, int(w.N * budget / (full * (args.steps + args.warmup))))
        for _ in range(args.warmup):
            oracle_step(oracle, src, nrows, prm, pool, threads)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            oracle_step(oracle, src, nrows, prm, pool, threads)
        el = time.perf_counter() - t0
    value = nrows * w.T * args.steps / el
    sample = ("%d of %d rows x T=%d per step, all seven estimators, float64 C oracle on %d "
              "threads" % (nrows, w.N, w.T, threads))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "num_envs": w.N, "seq_len": w.T, "estimators": 7,
                   "rows_per_step": nrows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def make_sets(torch, rl, src, dev, nsets, ests):
    """nsets independent device copies of every estimator's inputs and outputs."""
    sets = []
    for _ in range(nsets):
        st = {}
        for est in ests:
            ins, outs = SPECS[est]
            e = {k: torch.from_numpy(src[k]).to(dev) for k in ins + ("bootstrap_value",)}
            odt = torch.int32 if base_name(est) == "episodic_prefix_sum" else torch.float32
            for o in outs:
                e[o] = torch.empty(e[ins[0]].shape, dtype=odt, device=dev)
            st[est] = e
        sets.append(st)
    return sets


def launch(rl, est, e, prm):
    g, lm = prm["gamma"], prm["lambda_"]
    base = base_name(est)
    # the time-major entry point of the same estimator, else the row-major one
    f = getattr(rl, "rlcs_" + (est if est.endswith("_tm") else base))
    tr = {k: e[k] for k in TRUNC_IN if k in e}
    if base == "gae":
        f(e["rewards"], e["values"], e["terminateds"], g, lm, e["bootstrap_value"], out=e["out"],
          **tr)
    elif base == "lambda_returns":
        f(e["rewards"], e["values"], e["terminateds"], g, lm, e["bootstrap_value"], out=e["out"],
          **tr)
    elif base == "discounted_returns":
        f(e["rewards"], e["terminateds"], g, e["bootstrap_value"], out=e["out"], **tr)
    elif base == "vtrace":
        f(e["rewards"], e["values"], e["log_rhos"], e["terminateds"], g, lm, prm["rho_bar"],
          prm["c_bar"], e["bootstrap_value"], out=e["vs"], out_pg=e["pg"], **tr)
    elif base == "retrace":
        f(e["rewards"], e["values"], e["q_values"], e["log_rhos"], e["terminateds"], g, lm,
          prm["c_bar"], e["bootstrap_value"], out=e["out"], **tr)
    elif base == "eligibility_traces":
        f(e["x"], e["terminateds"], g, lm, out=e["out"])
    elif base == "episodic_prefix_sum":
        f(e["x_int"], e["terminateds"], out=e["out"])
    elif base == "gae_and_returns":
        f(e["rewards"], e["values"], e["terminateds"], g, lm, e["bootstrap_value"], out=e["out"],
          out_returns=e["out2"])
    elif base == "affine_scan":
        f(e["a"], e["b"], e["reset"], e["x_init"], reverse=True, out=e["out"])
    elif base == "gae_compact":
        f(e["rewards_bf16"], e["values_bf16"], e["terminateds_u8"], g, lm, e["bootstrap_value"],
          out=e["out"])
    else:
        raise ValueError(est)


def group_kwargs(est, e, prm):
    """Keyword arguments of rlcs_run_group for one estimator's buffer set."""
    g, lm = prm["gamma"], prm["lambda_"]
    tr = {k: e[k] for k in TRUNC_IN if k in e}
    base = base_name(est)
    if base in ("gae", "lambda_returns"):
        return dict(rewards=e["rewards"], values=e["values"], terminateds=e["terminateds"],
                    gamma=g, lambda_=lm, bootstrap_value=e["bootstrap_value"], out=e["out"], **tr)
    if base == "discounted_returns":
        return dict(rewards=e["rewards"], terminateds=e["terminateds"], gamma=g,
                    bootstrap_value=e["bootstrap_value"], out=e["out"], **tr)
    if base == "vtrace":
        return dict(rewards=e["rewards"], values=e["values"], log_rhos=e["log_rhos"],
                    terminateds=e["terminateds"], gamma=g, lambda_=lm, rho_bar=prm["rho_bar"],
                    c_bar=prm["c_bar"], bootstrap_value=e["bootstrap_value"], out=e["vs"],
                    out_pg=e["pg"], **tr)
    if base == "retrace":
        return dict(rewards=e["rewards"], values=e["values"], q_values=e["q_values"],
                    log_rhos=e["log_rhos"], terminateds=e["terminateds"], gamma=g, lambda_=lm,
                    c_bar=prm["c_bar"], bootstrap_value=e["bootstrap_value"], out=e["out"], **tr)
    if base == "eligibility_traces":
        return dict(x=e["x"], dones=e["terminateds"], gamma=g, lambda_=lm, out=e["out"])
    if base == "episodic_prefix_sum":
        return dict(x=e["x_int"], dones=e["terminateds"], out=e["out"])
    raise ValueError(est)


def capture(torch, stream, fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def time_graph(torch, stream, graph, reps):
    """Seconds for `reps` replays; replay() launches on the current stream, so
    the replays and both events go to `stream`."""
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(reps):
            graph.replay()
        end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / 1e3


def time_graph_each(torch, stream, graph, reps):
    """Seconds of each of `reps` back-to-back replays (an event between
    consecutive replays, all on `stream`)."""
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for i in range(reps):
            graph.replay()
            evs[i + 1].record(stream)
    evs[-1].synchronize()
    return [evs[i].elapsed_time(evs[i + 1]) / 1e3 for i in range(reps)]


def percentile(xs, q):
    ys = sorted(xs)
    return ys[min(len(ys) - 1, max(0, int(round(q * (len(ys) - 1)))))]


def replay_plan(n, block):
    """n steps as (rem, full): one graph of rem steps, then full replays of a
    graph of `block` steps (rem first, so that every later graph starts on
    the rotating set after the one the previous graph ended on)."""
    return n % block, n // block


def headline_line(value, ms_per_step, steps, warmup, n_gpus, config, step_gbs, peak, roofline,
                  cpu, e2e, launches, clocks, detail_path):
    """The one JSON line the bench prints: the headline and the objects the
    report needs, a few hundred bytes (the per-estimator and sweep figures go
    to the detail file)."""
    def r(x, nd=4):
        return None if x is None else float("%.*g" % (nd, x))
    line = {
        "metric": METRIC, "value": r(value, 6), "unit": UNIT, "n_gpus": n_gpus,
        "steps": steps, "warmup": warmup, "ms_per_step": r(ms_per_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": config,
        "hbm_gbs": r(step_gbs), "hbm_frac_of_8tbs": r(step_gbs / NOMINAL_HBM_GBS),
        "hbm_frac_of_measured": r(step_gbs / peak),
        "roofline": {k: (r(v) if isinstance(v, float) else v) for k, v in roofline.items()},
        "cpu_baseline": None if cpu is None else {
            "value": r(cpu["value"]), "unit": cpu["unit"], "cores": cpu["cores"],
            "kind": cpu["kind"], "sample": cpu["sample"]},
        "e2e": {"value": r(e2e["value"]), "unit": e2e["unit"],
                "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
                "d2h_bytes_per_step": e2e["d2h_bytes_per_step"]},
        "gpu_launches": launches,
        "clocks": {"sm_mhz": clocks.get("sm_mhz"), "sm_max_mhz": clocks.get("sm_max_mhz"),
                   "reasons": clocks.get("reasons", [])},
        "detail": detail_path,
    }
    return json.dumps(line, separators=(",", ":"))


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    dist = init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import linear_recurrence_scan_affine_gb300 as rl

    w = WORKLOADS[WORKLOAD]
    N, T = w.N, w.T
    prm = dict(gamma=w.gamma, lambda_=w.lambda_, rho_bar=w.rho_bar, c_bar=w.c_bar)
    src = rollout(N, T, w.seed + rank, w.p_term)
    order = list(ESTIMATORS)
    sets = make_sets(torch, rl, src, dev, ROTATING_SETS, order)
    footprint = sum(t.numel() * t.element_size() for st in sets for e in st.values()
                    for t in e.values())
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    stream = torch.cuda.Stream(dev)
    # One side stream per estimator: the seven calls of a step are independent,
    # so this schedule lets their fixed per-launch latencies overlap.
    side = {est: torch.cuda.Stream(dev) for est in order}

    def one_step(i):
        st = sets[i % ROTATING_SETS]
        if args.schedule == "grouped":
            rl.rlcs_run_group([(est, group_kwargs(est, st[est], prm)) for est in order])
        else:
            for est in order:
                launch(rl, est, st[est], prm)

    def steps_fn(n, start):
        """Steps start .. start+n-1 (buffer set i % ROTATING_SETS for step i)."""
        def fn():
            if args.schedule == "streams":
                for est in order:
                    side[est].wait_stream(stream)
                    with torch.cuda.stream(side[est]):
                        for i in range(start, start + n):
                            launch(rl, est, sets[i % ROTATING_SETS][est], prm)
                for est in order:
                    stream.wait_stream(side[est])
            else:
                for i in range(start, start + n):
                    one_step(i)
        return fn

    # Set-up, not steps: one eager call of each estimator on every stream the
    # graphs use (loads the kernels, creates any workspace outside capture).
    for s_ in [stream] + list(side.values()):
        s_.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s_):
            one_step(0)
    torch.cuda.synchronize()
    rl.check_all_workspaces()

    # graphs of whole steps; K and W are met exactly by a remainder graph
    # plus replays of a BLOCK-step graph
    BLOCK = 8 * ROTATING_SETS
    K, W = max(1, args.steps), max(0, args.warmup)
    graphs = {}

    def graph(n, start):
        key = (n, start % ROTATING_SETS)
        if key not in graphs:
            graphs[key] = capture(torch, stream, steps_fn(n, key[1]))
        return graphs[key]

    def sequence(n, cursor):
        rem, full = replay_plan(n, BLOCK)
        seq = []
        if rem:
            seq.append(graph(rem, cursor))
            cursor += rem
        seq += [graph(BLOCK, cursor)] * full
        return seq, cursor + full * BLOCK

    warm_seq, cursor = sequence(W, 0)
    timed_seq, _ = sequence(K, cursor)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for g_ in warm_seq:
            g_.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(dev.index if "CUDA_VISIBLE_DEVICES" not in os.environ
                           else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]))
    sampler.start()
    time.sleep(0.3)  # let the sampler take its first reading
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        # a ~1 ms device-side delay ahead of the start event: the host queues
        # every replay meanwhile, so the timed region holds device work only
        torch.cuda._sleep(2_000_000)
        t_start.record(stream)
        for g_ in timed_seq:
            g_.replay()
        t_end.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop()
    elapsed = t_start.elapsed_time(t_end) / 1e3
    elapsed = max_over_ranks(dist, elapsed, dev)
    rl.check_all_workspaces()
    del graphs, warm_seq, timed_seq

    step_bytes = sum(bytes_per_launch(e, N, T) for e in order)
    value = world * N * T * K / elapsed
    step_gbs = step_bytes * K / elapsed / 1e9

    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            peaks = json.load(fh)
    except (OSError, ValueError):
        pass
    peak = peaks.get("hbm_gbs")
    peak_src = "measured hbm_gbs (copy burst)"
    if not peak:
        peak, peak_src = 6800.0, "fallback 6.8 TB/s"

    # every estimator alone: a graph of back-to-back launches, each on its own
    # buffer set, with enough sets that the rotation spans >= 3x the L2
    per_est = {est: time_alone(torch, rl, est, src, dev, stream, prm, l2, N, T) for est in order}
    for r_ in per_est.values():
        r_["frac_of_measured_hbm"] = r_["gbs"] / peak
    # the dominant kernel: the slowest estimator alone
    dom = max(per_est, key=lambda e: per_est[e]["us_per_launch"])
    dom_bytes = bytes_per_launch(dom, N, T)
    dom_us = per_est[dom]["us_per_launch"]
    traffic = None
    tr_path = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tr_path):
        with open(tr_path) as fh:
            tr = json.load(fh)
        # counters count only for the kernel sources they were taken on
        if tr.get("kernel_source_sha256_16") == kernel_source_hash():
            traffic = tr.get("%s_%dx%d" % (dom, N, T))
    achieved = dom_bytes / (dom_us * 1e-6) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic, "kernel": dom,
                "bytes_per_launch": dom_bytes, "us_per_launch": dom_us,
                "peak_source": peak_src}
    detail = {"per_estimator_4096x128": per_est,
              "roofline": dict(roofline, timing=(
                  "kernel alone: CUDA graph of back-to-back launches, each on its own buffer "
                  "set (rotation >= 3x L2), CUDA events on the launching stream; >= 20 "
                  "replays"))}
    # what any launch of this size and shape costs: the diagnostic copy of the
    # same bytes, and the same grid doing nothing
    n_arrays = len(SPECS[dom][0]) + len(SPECS[dom][1])
    copy_us = time_diag(torch, rl, n_arrays, dev, stream, l2, N, T, False)
    empty_us = time_diag(torch, rl, n_arrays, dev, stream, l2, N, T, True)
    detail["roofline"]["reference"] = {
        "stream_copy_us": copy_us, "empty_launch_us": empty_us,
        "stream_copy_frac": dom_bytes / (copy_us * 1e-6) / 1e9 / peak,
        "kernel_over_copy": dom_us / copy_us,
        "what": "rlcs_diag_stream_copy: the warp-row launch shape moving the same bytes "
                "(%d arrays x %d rows x %d steps) with no scan (same prefetch and programmatic "
                "dependent launch); empty = the same grid that only waits and exits"
                % (n_arrays, N, T)}
    # the same step in every schedule
    detail["schedules_4096x128"] = time_step(torch, rl, order, src, dev, stream, prm, l2, N, T)

    # GAE alone at 64 x 512, and the five truncated estimators at 4096 x 128
    w1 = WORKLOADS["gae_64x512"]
    src1 = rollout(w1.N, w1.T, w1.seed, w1.p_term)
    prm1 = dict(gamma=w1.gamma, lambda_=w1.lambda_, rho_bar=w1.rho_bar, c_bar=w1.c_bar)
    r_ = time_alone(torch, rl, "gae", src1, dev, stream, prm1, l2, w1.N, w1.T)
    r_["frac_of_measured_hbm"] = r_["gbs"] / peak
    detail["gae_64x512"] = r_
    w3 = WORKLOADS["trunc5_4096x128"]
    src3 = rollout(w3.N, w3.T, w3.seed, w3.p_term, w3.p_trunc)
    prm3 = dict(gamma=w3.gamma, lambda_=w3.lambda_, rho_bar=w3.rho_bar, c_bar=w3.c_bar)
    ests3 = [e + "_trunc" for e in w3.estimators]
    res3 = {}
    for est in ests3:
        r_ = time_alone(torch, rl, est, src3, dev, stream, prm3, l2, w3.N, w3.T)
        r_["frac_of_measured_hbm"] = r_["gbs"] / peak
        res3[est] = r_
    step3 = time_step(torch, rl, ests3, src3, dev, stream, prm3, l2, w3.N, w3.T)
    step3["frac_of_measured_hbm"] = step3["gbs"] / peak
    detail["trunc5_4096x128"] = {"alone": res3, "step": step3}
    del src1, src3

    # the long-row recipes, every estimator alone (same method as above)
    if not args.no_long_t:
        # SM clocks over each section, beside its numbers (later sections run
        # after seconds of load and may see lower clocks than the headline)
        gpu_index = (dev.index if "CUDA_VISIBLE_DEVICES" not in os.environ
                     else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]))
        sect_clock = ClockSampler(gpu_index)
        sect_clock.start()
        long_t = {}
        for name in ("longT_256x1024", "longT_256x4096", "longT_256x16384", "vlong_8x131072"):
            wl = WORKLOADS[name]
            prm_l = dict(gamma=wl.gamma, lambda_=wl.lambda_, rho_bar=wl.rho_bar, c_bar=wl.c_bar)
            src_l = rollout(wl.N, wl.T, wl.seed, wl.p_term)
            res = {}
            for est in wl.estimators:
                r_ = time_alone(torch, rl, est, src_l, dev, stream, prm_l, l2, wl.N, wl.T,
                                seconds=0.08)
                r_["frac_of_measured_hbm"] = r_["gbs"] / peak
                res[est] = r_
            step_l = time_step(torch, rl, wl.estimators, src_l, dev, stream, prm_l, l2, wl.N,
                               wl.T)
            step_l["frac_of_measured_hbm"] = step_l["gbs"] / peak
            long_t[name] = {"step": step_l, "alone": res}
            del src_l
        rl.check_all_workspaces()
        long_t["clocks"] = sect_clock.stop()
        detail["long_t_sweep"] = long_t

        # entry points beyond the seven, alone, at the bench size and one long
        # size; fp32 GAE on the same data is timed beside compact GAE
        from synthetic_rollouts import affine_inputs, compact_rollout
        sect_clock = ClockSampler(gpu_index)
        sect_clock.start()
        next_rows = {}
        for (nN, nT, seed) in ((N, T, w.seed), (256, 16384, 1004)):
            srcn = dict(rollout(nN, nT, seed, w.p_term), **affine_inputs(nN, nT, seed + 7))
            comp, _ = compact_rollout(nN, nT, seed + 9, w.p_term)
            srcn.update(rewards_bf16=comp["rewards"], values_bf16=comp["values"],
                        terminateds_u8=comp["terminateds"])
            # the same arrays stored time-major for the _tm entry points
            srcn_tm = {k: (np.ascontiguousarray(v.T) if v.ndim == 2 else v)
                       for k, v in srcn.items()}
            res = {}
            for est in EXTRA:
                if est == "gae_compact":
                    r_ = time_alone(torch, rl, "gae", srcn, dev, stream, prm, l2, nN, nT,
                                    seconds=0.08)
                    r_["frac_of_measured_hbm"] = r_["gbs"] / peak
                    res["gae_fp32_same_data"] = r_
                r_ = time_alone(torch, rl, est, srcn_tm if est.endswith("_tm") else srcn, dev,
                                stream, prm, l2, nN, nT, seconds=0.08)
                r_["frac_of_measured_hbm"] = r_["gbs"] / peak
                res[est] = r_
            next_rows["%dx%d" % (nN, nT)] = res
            del srcn, srcn_tm
        rl.check_all_workspaces()
        next_rows["clocks"] = sect_clock.stop()
        detail["next_rows"] = next_rows

        # the seven time-major entry points at three more sizes: 8-environment
        # chunks in one block per SM (256 x 4096) and in one partial wave
        # (8 x 131072), and 32-environment chunks (1024 x 4096)
        sect_clock = ClockSampler(gpu_index)
        sect_clock.start()
        tm_sizes = {}
        for (nN, nT, seed) in ((256, 4096, 1004), (8, 131072, 1004), (1024, 4096, 1004)):
            srcn_tm = {k: (np.ascontiguousarray(v.T) if v.ndim == 2 else v)
                       for k, v in rollout(nN, nT, seed, w.p_term).items()}
            res = {}
            for est in ESTIMATORS:
                r_ = time_alone(torch, rl, est + "_tm", srcn_tm, dev, stream, prm, l2, nN, nT,
                                seconds=0.08)
                r_["frac_of_measured_hbm"] = r_["gbs"] / peak
                res[est + "_tm"] = r_
            tm_sizes["%dx%d" % (nN, nT)] = res
            del srcn_tm
        rl.check_all_workspaces()
        tm_sizes["clocks"] = sect_clock.stop()
        detail["time_major_sizes"] = tm_sizes

    e2e = run_e2e(torch, rl, src, dev, stream, prm, order, max(32, min(K, 512)), N, T)
    e2e["value"] *= world
    detail["e2e"] = e2e

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = time_oracle(src, prm, budget_s=args.cpu_seconds)
        detail["cpu_baseline"] = cpu

    if rank == 0:
        launches = (1 if args.schedule == "grouped" else len(order)) * K
        launch_desc = {
            "streams": "seven rlcs_* calls per step on seven streams (fork/join per graph)",
            "serial": "seven rlcs_* calls per step on one stream",
            "grouped": "one rlcs_run_group call per step (the seven in one launch)"}
        config = {"workload": WORKLOAD, "num_envs": N, "seq_len": T, "estimators": 7,
                  "bytes_per_step": step_bytes,
                  "l2": "inputs larger than L2: %d rotating buffer sets, %.0f MB = %.1fx L2"
                        % (ROTATING_SETS, footprint / 1e6, footprint / l2),
                  "launch": launch_desc[args.schedule] + "; CUDA graphs of whole steps",
                  "parallelism": "weak: each rank its own batch"}
        detail["headline"] = {"schedule": args.schedule, "steps": K, "warmup": W,
                              "elapsed_s": elapsed, "clocks": clocks, "config": config}
        detail["kernel_source_sha256_16"] = kernel_source_hash()
        detail_path = args.detail
        try:
            d = os.path.dirname(os.path.abspath(detail_path))
            os.makedirs(d, exist_ok=True)
            with open(detail_path, "w") as fh:
                json.dump(detail, fh, indent=1)
        except OSError as exc:
            detail_path = "not written: %s" % exc
        print(headline_line(value, 1e3 * elapsed / K, K, W, world, config, step_gbs, peak,
                            roofline, cpu, e2e, launches, clocks, detail_path), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def time_alone(torch, rl, est, src, dev, stream, prm, l2, N, T, seconds=0.15):
    ins, outs = SPECS[est]
    row_key = "x_init" if est == "affine_scan" else "bootstrap_value"
    set_bytes = bytes_per_launch(est, N, T)
    nsets = int(min(256, max(8, -(-3 * l2 // set_bytes))))
    sets = []
    for _ in range(nsets):
        e = {k: torch.from_numpy(src[k]).to(dev) for k in ins + (row_key,)}
        odt = torch.int32 if est.startswith("episodic_prefix_sum") else torch.float32
        for o in outs:
            e[o] = torch.empty(e[ins[0]].shape, dtype=odt, device=dev)
        sets.append(e)
    with torch.cuda.stream(stream):
        for e in sets:
            launch(rl, est, e, prm)
    torch.cuda.synchronize()
    g = capture(torch, stream, lambda: [launch(rl, est, e, prm) for e in sets])
    with torch.cuda.stream(stream):
        g.replay()
    once = time_graph(torch, stream, g, 1)
    reps = max(20, int(seconds / max(1e-6, once)))
    # throughput from one continuous timed region; the spread from the same
    # number of replays timed one by one (an event between replays breaks
    # the launch overlap from one replay into the next, which adds about
    # 2 us per replay, so those run slightly slower)
    sec = time_graph(torch, stream, g, reps) / (reps * nsets)
    each = [t / nsets for t in time_graph_each(torch, stream, g, reps)]
    # cold: one call after a write of 3x the L2 has flushed it (event timing)
    flush = torch.empty(3 * l2, dtype=torch.uint8, device=dev)
    cold = []
    for i in range(3):
        with torch.cuda.stream(stream):
            flush.fill_(i)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            launch(rl, est, sets[i % nsets], prm)
            b.record(stream)
        b.synchronize()
        cold.append(a.elapsed_time(b) / 1e3)
    del g, sets, flush
    torch.cuda.synchronize()
    torch.cuda.empty_cache()  # the next measurement allocates afresh
    return {"us_per_launch": sec * 1e6, "us_median_of_replays": percentile(each, 0.5) * 1e6,
            "us_p10": percentile(each, 0.1) * 1e6, "us_p90": percentile(each, 0.9) * 1e6,
            "replays": reps,
            "us_cold_single_call": percentile(cold, 0.5) * 1e6,
            "env_steps_per_s": N * T / sec,
            "gbs": bytes_per_launch(est, N, T) / sec / 1e9,
            "bytes_per_env_step": bytes_per_env_step(est), "rotating_sets": nsets,
            "footprint_over_l2": nsets * set_bytes / l2,
            "timing": "mean over one timed region of graph replays of back-to-back launches, "
                      "one per rotating buffer set; median, p10, p90 of the replays timed one "
                      "by one; cold = one call after an L2 flush"}


def time_step(torch, rl, ests, src, dev, stream, prm, l2, N, T, seconds=0.15):
    """The estimators of one step over rotating buffer sets that span >= 3x
    the L2, in several schedules: each estimator on its own stream (as the
    headline step), all on one stream, one rlcs_run_group call, and the
    estimators split into 2 or 3 groups, each group's call on its own
    stream. Returns all of them and, as the step, the fastest: time per step
    and the step's algorithmic GB/s."""
    step_bytes = sum(bytes_per_launch(e, N, T) for e in ests)
    nsets = int(min(64, max(2, -(-3 * l2 // step_bytes))))
    sets = make_sets(torch, rl, src, dev, nsets, ests)
    side = {est: torch.cuda.Stream(dev) for est in ests}
    for est in ests:  # warm-up: every side stream's workspace exists before capture
        side[est].wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side[est]):
            for st in sets:
                launch(rl, est, st[est], prm)
    torch.cuda.synchronize()

    def concurrent():
        for est in ests:
            side[est].wait_stream(stream)
            with torch.cuda.stream(side[est]):
                for st in sets:
                    launch(rl, est, st[est], prm)
        for est in ests:
            stream.wait_stream(side[est])

    def serial():
        for st in sets:
            for est in ests:
                launch(rl, est, st[est], prm)

    group_calls = [[(base_name(est), group_kwargs(est, st[est], prm)) for est in ests]
                   for st in sets]

    def grouped():
        for calls in group_calls:
            rl.rlcs_run_group(calls)

    # k groups, each one rlcs_run_group call per buffer set on its own stream
    # (estimators dealt round-robin, heaviest first)
    order = sorted(ests, key=lambda e: -bytes_per_launch(e, N, T))
    split = {k: [order[i::k] for i in range(k)] for k in (2, 3) if len(ests) > k}
    gside = {k: [torch.cuda.Stream(dev) for _ in range(k)] for k in split}

    def groups_on_streams(k):
        def run():
            for part, s in zip(split[k], gside[k]):
                s.wait_stream(stream)
                with torch.cuda.stream(s):
                    for st in sets:
                        rl.rlcs_run_group([(base_name(e), group_kwargs(e, st[e], prm))
                                           for e in part])
            for s in gside[k]:
                stream.wait_stream(s)
        return run

    with torch.cuda.stream(stream):  # the one-stream schedules' workspaces
        serial()
        grouped()
    for k in split:  # and the group streams' (created before capture)
        groups_on_streams(k)()
    torch.cuda.synchronize()
    us = {}
    schedules = [("streams", concurrent), ("one_stream", serial), ("grouped", grouped)]
    schedules += [("groups_on_%d_streams" % k, groups_on_streams(k)) for k in split]
    for name, fn in schedules:
        g = capture(torch, stream, fn)
        with torch.cuda.stream(stream):
            g.replay()
        once = time_graph(torch, stream, g, 1)
        reps = max(3, int(seconds / max(1e-6, once)))
        us[name] = time_graph(torch, stream, g, reps) / (reps * nsets) * 1e6
        del g
    del sets
    torch.cuda.synchronize()
    best = min(us, key=us.get)
    sec = us[best] * 1e-6
    return {"us_per_step": us[best], "schedule": best,
            "us_per_step_by_schedule": us, "env_steps_per_s": N * T / sec,
            "gbs": step_bytes / sec / 1e9, "bytes_per_step": step_bytes,
            "estimators": list(ests), "rotating_sets": nsets,
            "footprint_over_l2": nsets * step_bytes / l2}


def time_diag(torch, rl, n_arrays, dev, stream, l2, N, T, empty, seconds=0.1):
    """The library's diagnostic stream copy in the warp-row launch shape:
    n_arrays - 1 inputs summed into one output (the same bytes per launch as
    an estimator with n_arrays arrays), back to back on rotating buffers; with
    `empty` the same grid only waits and exits. Returns us per launch."""
    n_in = max(1, n_arrays - 1)
    set_bytes = n_arrays * N * T * 4
    nsets = int(min(256, max(8, -(-3 * l2 // set_bytes))))
    sets = [([torch.zeros(N, T, device=dev) for _ in range(n_in)], torch.empty(N, T, device=dev))
            for _ in range(nsets)]
    with torch.cuda.stream(stream):
        for ins, out in sets:
            rl.rlcs_diag_stream_copy(ins, out, empty)
    torch.cuda.synchronize()
    g = capture(torch, stream, lambda: [rl.rlcs_diag_stream_copy(i, o, empty) for i, o in sets])
    with torch.cuda.stream(stream):
        g.replay()
    once = time_graph(torch, stream, g, 1)
    reps = max(3, int(seconds / max(1e-6, once)))
    sec = time_graph(torch, stream, g, reps) / (reps * nsets)
    del g, sets
    torch.cuda.synchronize()
    return sec * 1e6


def run_e2e(torch, rl, src, dev, stream, prm, order, steps, N, T, depth=2, block=16):
    """Whole steps through the public API from pinned host memory.

    Like a rollout buffer, one step's rollout (every array any of the seven
    estimators reads, each once: rewards, values, terminateds, log_rhos,
    q_values, x, x_int and the bootstrap values) sits in one contiguous pinned
    host buffer and the outputs come back into another. Each step copies the
    rollout in with one host-to-device copy, runs the seven rlcs_* calls on
    it, and copies every output back with one device-to-host copy. Steps are
    pipelined over `depth` device buffer slots on separate copy-in, compute
    and copy-out streams, so step i+1's copy-in overlaps step i's kernels and
    step i-1's copy-out."""
    in_names = []
    for est in order:
        for k in ESTIMATORS[est][0] + ("bootstrap_value",):
            if k not in in_names:
                in_names.append(k)

    def place(items):
        off, fields = 0, []
        for key, ref in items:
            fields.append((key, off, ref.shape, ref.dtype))
            off += (ref.size * ref.itemsize + 255) // 256 * 256
        return fields, off

    in_fields, in_bytes = place([(k, src[k]) for k in in_names])
    out_fields, out_bytes = place([((est, o), src["rewards"]) for est in order
                                   for o in ESTIMATORS[est][1]])
    h_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    for k, off, shp, dt in in_fields:
        a = src[k]
        h_in[off:off + a.size * a.itemsize].copy_(torch.from_numpy(a.view(np.uint8).reshape(-1)))
    h_out = [torch.empty(out_bytes, dtype=torch.uint8).pin_memory() for _ in range(depth)]
    d_in = [torch.empty(in_bytes, dtype=torch.uint8, device=dev) for _ in range(depth)]
    d_out = [torch.empty(out_bytes, dtype=torch.uint8, device=dev) for _ in range(depth)]
    tdt = {np.dtype(np.float32): torch.float32, np.dtype(np.int32): torch.int32}

    def views(buf_in, buf_out):
        shared = {}
        for k, off, shp, dt in in_fields:
            n = int(np.prod(shp))
            shared[k] = buf_in[off:off + n * 4].view(tdt[dt]).view(*shp)
        sets = {est: {k: shared[k] for k in ESTIMATORS[est][0] + ("bootstrap_value",)}
                for est in order}
        for (est, k), off, shp, dt in out_fields:
            n = int(np.prod(shp))
            ref_dt = tdt[src[ESTIMATORS[est][0][0]].dtype]
            sets[est][k] = buf_out[off:off + n * 4].view(ref_dt).view(*shp)
        return sets

    slot_sets = [views(d_in[i], d_out[i]) for i in range(depth)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    side = {est: torch.cuda.Stream(dev) for est in order}

    def step(i, slot, ev):
        # copy-in may reuse the slot once the kernels of step i - depth are done
        if ev["comp"][slot] is not None:
            s_in.wait_event(ev["comp"][slot])
        with torch.cuda.stream(s_in):
            d_in[slot].copy_(h_in, non_blocking=True)
        e_in = torch.cuda.Event()
        e_in.record(s_in)
        joins = []
        for est in order:
            st = side[est]
            st.wait_event(e_in)
            if ev["out"][slot] is not None:   # outputs of step i - depth copied out
                st.wait_event(ev["out"][slot])
            with torch.cuda.stream(st):
                launch(rl, est, slot_sets[slot][est], prm)
            e = torch.cuda.Event()
            e.record(st)
            joins.append(e)
        for e in joins:
            s_out.wait_event(e)
        e_comp = torch.cuda.Event()
        e_comp.record(s_out)
        with torch.cuda.stream(s_out):
            h_out[slot].copy_(d_out[slot], non_blocking=True)
        e_out = torch.cuda.Event()
        e_out.record(s_out)
        ev["comp"][slot], ev["out"][slot] = e_comp, e_out

    def block_fn():
        ev = {"comp": [None] * depth, "out": [None] * depth}
        for s_ in [s_in, s_out] + list(side.values()):
            s_.wait_stream(stream)
        for i in range(block):
            step(i, i % depth, ev)
        for s_ in [s_in, s_out] + list(side.values()):
            stream.wait_stream(s_)

    with torch.cuda.stream(stream):
        block_fn()  # eager warm-up: workspaces allocated outside capture
    torch.cuda.synchronize()
    g = capture(torch, stream, block_fn)
    with torch.cuda.stream(stream):
        for _ in range(2):
            g.replay()
    reps = max(2, -(-steps // block))
    sec = time_graph(torch, stream, g, reps) / (reps * block)
    return {"value": N * T / sec, "unit": UNIT, "h2d_bytes_per_step": in_bytes,
            "d2h_bytes_per_step": out_bytes, "ms_per_step": sec * 1e3,
            "h2d_gbs": in_bytes / sec / 1e9, "d2h_gbs": out_bytes / sec / 1e9,
            "path": "one pinned host->device copy of the rollout (each array the seven "
                    "estimators read, once), seven rlcs_* calls on seven streams, one "
                    "device->pinned host copy of all outputs, per step; %d-slot pipeline over "
                    "copy-in / compute / copy-out streams, CUDA graph of %d steps"
                    % (depth, block)}


def run_profile(args):
    """Eager launches of one estimator on rotating buffer sets (no graphs, no
    timing): a small, fixed launch sequence for ncu captures."""
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import linear_recurrence_scan_affine_gb300 as rl
    w = WORKLOADS[args.workload]
    N = args.rows or w.N
    prm = dict(gamma=w.gamma, lambda_=w.lambda_, rho_bar=w.rho_bar, c_bar=w.c_bar)
    est = args.profile
    p_trunc = (w.p_trunc or 0.005) if est.endswith("_trunc") else 0.0
    src = rollout(N, w.T, w.seed, w.p_term, p_trunc)
    if est == "group":  # the workload's estimators as one rlcs_run_group call
        nsets = max(2, min(ROTATING_SETS, args.sets))
        sets = []
        for _ in range(nsets):
            st = {}
            for e_ in w.estimators:
                ins, outs = ESTIMATORS[e_]
                e = {k: torch.from_numpy(src[k]).to(dev) for k in ins + ("bootstrap_value",)}
                for o in outs:
                    e[o] = torch.empty(e[ins[0]].shape, device=dev,
                                       dtype=torch.int32 if e_ == "episodic_prefix_sum"
                                       else torch.float32)
                st[e_] = e
            sets.append([(e_, group_kwargs(e_, st[e_], prm)) for e_ in w.estimators])
        for i in range(args.warmup + args.steps):
            rl.rlcs_run_group(sets[i % nsets])
        torch.cuda.synchronize()
        rl.check_all_workspaces()
        print(json.dumps({"profile": "group", "workload": args.workload, "N": N, "T": w.T,
                          "launches": args.warmup + args.steps,
                          "bytes_per_launch": sum(bytes_per_launch(e_, N, w.T)
                                                  for e_ in w.estimators)}))
        return 0
    if est in EXTRA:  # the extra entry points' own inputs, drawn as in next_rows
        from synthetic_rollouts import affine_inputs, compact_rollout
        src.update(affine_inputs(N, w.T, w.seed + 7))
        comp, _ = compact_rollout(N, w.T, w.seed + 9, w.p_term)
        src.update(rewards_bf16=comp["rewards"], values_bf16=comp["values"],
                   terminateds_u8=comp["terminateds"])
    if est.endswith("_tm"):  # the same arrays stored time-major
        src = {k: (np.ascontiguousarray(v.T) if v.ndim == 2 else v) for k, v in src.items()}
    nsets = max(2, min(ROTATING_SETS, args.sets))
    sets = []
    row_key = "x_init" if est == "affine_scan" else "bootstrap_value"
    for _ in range(nsets):
        ins, outs = SPECS[est]
        e = {k: torch.from_numpy(src[k]).to(dev) for k in ins + (row_key,)}
        odt = torch.int32 if est.startswith("episodic_prefix_sum") else torch.float32
        for o in outs:
            e[o] = torch.empty(e[ins[0]].shape, dtype=odt, device=dev)
        sets.append(e)
    for i in range(args.warmup + args.steps):
        launch(rl, est, sets[i % nsets], prm)
    torch.cuda.synchronize()
    rl.check_all_workspaces()
    print(json.dumps({"profile": est, "workload": args.workload, "N": N, "T": w.T,
                      "launches": args.warmup + args.steps,
                      "bytes_per_launch": bytes_per_launch(est, N, w.T)}))
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-long-t", action="store_true",
                    help="skip the long-row sweep, the extra entry points and the time-major sizes")
    ap.add_argument("--schedule", choices=("streams", "serial", "grouped"), default="streams",
                    help="how the headline step issues its seven calls")
    ap.add_argument("--detail", default="bench_detail.json",
                    help="where to write the per-estimator and sweep figures (JSON)")
    ap.add_argument("--profile", choices=tuple(SPECS) + ("group",), default=None,
                    help="eager launches of one estimator only (for ncu)")
    ap.add_argument("--workload", default=WORKLOAD, choices=tuple(WORKLOADS))
    ap.add_argument("--rows", type=int, default=0, help="profile mode: rows (0 = workload's N)")
    ap.add_argument("--sets", type=int, default=ROTATING_SETS)
    args = ap.parse_args()
    if args.profile:
        return run_profile(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
