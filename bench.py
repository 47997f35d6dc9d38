#!/usr/bin/env python
"""Benchmark of the finite-automaton constrained denoising step on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference] [--workload NAME]

One step = one fa_constrained_step call over one batch: emission reweighting, the span
up-sweep, root and top-down sampling with prefix/suffix messages, leaf tokens with
constrained marginals, and the top-k commit.  The default workload is the block-wise
decoding batch: a random DFA with 512 states (p_dead 0.9), vocabulary 151936, B=16
sequences of L=512 positions, all masked at the first step (synthetic, seeded); its whole
64-step block-wise remasking schedule is timed beside the step.  --workload picks another.

Timing: W untimed warm-up steps, then exactly K steps between a barrier and a device
synchronisation on both sides; each step is one CUDA-graph replay of the step, bracketed
by CUDA events on its stream, with a 256 MiB L2 flush between steps outside the events.
Stage boundaries are recorded inside the graph (fa_profile_enable), which gives the
per-stage device time used for the roofline of the dominant stage.  N > 1 runs
independent replicas (one per GPU, weak scaling); rank 0 prints one JSON line.

--impl reference times the float64 CPU oracle on the host cores on the same workload, a
bounded sample per step (the first sequences of the batch, as many as fit about 20 s).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ms per constrained denoising step and positions/s at 1 GB300; % of roofline"
UNIT = "positions/s"
DEFAULT_WORKLOAD = "blockwise_dfa_S512_L512"
FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-graph", action="store_true", help="launch the step eagerly instead of a graph replay")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-baseline sample budget")
    ap.add_argument("--e2e-steps", type=int, default=500)
    ap.add_argument("--length", type=int, default=None, help="override L (smaller profiling cases)")
    ap.add_argument("--method", default="tree", choices=["tree", "chain", "greedy"],
                    help="log-depth tree (default), the O(L) chain form of the same step, or greedy (T=0) "
                         "decoding by max-product over the tree")
    ap.add_argument("--schedule", dest="schedule", action="store_true", default=True,
                    help="also time the workload's whole remasking schedule (workloads with one; the default)")
    ap.add_argument("--no-schedule", dest="schedule", action="store_false",
                    help="skip the remasking schedule")
    ap.add_argument("--confidence", default="marginal", choices=["marginal", "neg_entropy", "unconstrained"],
                    help="remasking confidence the commit ranks by")
    return ap.parse_args()


# ----------------------------------------------------------------------------- distributed

def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(x, world):
    """Maximum of x over the ranks (the tensor lives where the process group's backend
    wants it: the GPU for nccl, the host for gloo)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(positions_per_rank, world, ms_max):
    """Whole-job throughput of independent replicas: every rank's positions over the
    slowest rank's step time."""
    return positions_per_rank * world / (ms_max / 1e3)


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks, power and throttle reasons sampled every 200 ms while running.

    Start it before the warm-up (wait_first() blocks until nvidia-smi answers), bracket the
    timed region with mark_start() / mark_end(), and summary() keeps the samples taken
    inside that window (all samples, flagged, if the window caught none)."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 200

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []          # (monotonic time, csv line)
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def wait_first(self, timeout: float = 10.0):
        end = time.monotonic() + timeout
        while self.proc is not None and not self.lines and time.monotonic() < end and self.proc.poll() is None:
            time.sleep(0.02)

    def mark_start(self):
        self.t0 = time.monotonic()

    def mark_end(self):
        # one more period so the sample covering the end of the region is read
        self.t1 = time.monotonic()
        time.sleep(self.PERIOD_MS / 1e3 + 0.05)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    @staticmethod
    def _parse(ln):
        f = [x.strip() for x in ln.split(",")]
        if len(f) < 9:
            return None
        try:
            sm, mx = float(f[1]), float(f[2])
        except ValueError:
            return None
        try:
            pw = float(f[3])
        except ValueError:
            pw = None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = [n for n, v in zip(names, f[5:9]) if v.lower().startswith("active")]
        return sm, mx, pw, reasons

    def summary(self):
        rows = [(t, self._parse(ln)) for t, ln in self.lines]
        rows = [(t, r) for t, r in rows if r is not None]
        if not rows:
            return None
        t0 = self.t0 if self.t0 is not None else -math.inf
        t1 = (self.t1 + self.PERIOD_MS / 1e3) if self.t1 is not None else math.inf
        inside = [r for t, r in rows if t0 <= t <= t1]
        use = inside if inside else [r for _, r in rows]
        sm = [r[0] for r in use]
        pw = [r[2] for r in use if r[2] is not None]
        reasons = sorted({n for r in use for n in r[3]})
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(r[1] for r in use)), "reasons": reasons,
                "samples": len(use), "samples_in_timed_region": len(inside),
                "power_w_median": float(np.median(pw)) if pw else None,
                "window_s": (self.t1 - self.t0) if (self.t0 is not None and self.t1 is not None) else None}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the CPU baseline."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model", "hardware")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


# ----------------------------------------------------------------------------- roofline model

def algorithmic(w, masked: int, method: str = "tree"):
    """Algorithmic bytes and FLOPs per step of each stage (the per-unit figures of the design
    notes times the units one step processes).  For the chain form the second and third
    stages are the forward pass and the backward pass with the state draws: each reads every
    M_t once and does one vector-matrix product per position."""
    B, L, S, V = w.B, w.L, w.S, w.V
    if method == "greedy":
        K = max(0, math.ceil(math.log2(L))) if L > 1 else 0
        nk = [(L + (1 << k) - 1) >> k for k in range(K + 1)]
        alg = algorithmic(w, masked, "tree")
        alg["upsweep"]["flops"] = 0          # max-product span products run on the CUDA cores
        alg["topdown"] = {"bytes": sum(B * n * 8 * S for n in nk[:K]), "flops": 0}  # two vectors per midpoint
        alg["leaf_commit"] = {"bytes": 4 * B * L * 2, "flops": 0}
        return alg
    if method == "chain":
        span = 4 * S * S + 8 * S
        msg = 8 * S
        return {"reweight": {"bytes": 4 * masked * V + B * L * span, "flops": 2 * masked * w.fa.n_incidences},
                "upsweep": {"bytes": B * L * (4 * S * S + msg), "flops": 2 * B * L * S * S},
                "topdown": {"bytes": B * L * (4 * S * S + 2 * msg), "flops": 2 * B * L * S * S},
                "leaf_commit": {"bytes": 4 * B * L * 4 + 8 * B * L, "flops": 0}}
    K = max(0, math.ceil(math.log2(L))) if L > 1 else 0
    nk = [(L + (1 << k) - 1) >> k for k in range(K + 1)]
    span = 4 * S * S + 8 * S                      # mantissas + row exponent + row max
    reweight = 4 * masked * V + B * L * span       # probs rows read once, leaf spans written
    products = sum(B * (nk[k - 1] // 2) for k in range(1, K + 1))   # real products (not copies)
    upsweep_bytes = sum(B * (nk[k - 1] + nk[k]) * span for k in range(1, K + 1))
    upsweep_flops = products * 2 * S ** 3
    topdown = sum(B * nk[k] * span for k in range(0, K))          # every non-root span read once
    return {"reweight": {"bytes": reweight, "flops": 2 * masked * w.fa.n_incidences},
            "upsweep": {"bytes": upsweep_bytes, "flops": upsweep_flops},
            "topdown": {"bytes": topdown, "flops": 2 * B * S * S * sum(nk[:K])},
            "leaf_commit": {"bytes": 4 * B * L * 4 + 8 * B * L, "flops": 0}}


def reweight_gather(w, masked: int, ms: float, clocks):
    """The reweight against its compute limits: one gather-add per token-edge incidence per
    masked position, against the FP32 issue peak (128 lanes per SM per clock) and the
    shared-memory gather peak (32 banks per SM per clock), at the sampled SM clock (152 SMs)."""
    if ms <= 0:
        return None
    mhz = (clocks or {}).get("sm_mhz") or 2070.0
    gathers = masked * w.fa.n_incidences
    rate = gathers / (ms / 1e3)
    alu = 152 * 128 * mhz * 1e6
    smem = 152 * 32 * mhz * 1e6
    return {"gathers": gathers, "achieved_G_per_s": rate / 1e9, "fp32_issue_peak_G_per_s": alu / 1e9,
            "frac_fp32_issue": rate / alu, "smem_gather_peak_G_per_s": smem / 1e9, "frac_smem_gather": rate / smem,
            "sm_mhz": mhz}


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def source_hash():
    h = hashlib.sha256()
    for f in sorted(os.listdir(os.path.join(ROOT, "constrained_decoding_diffusion_gb300", "csrc"))):
        with open(os.path.join(ROOT, "constrained_decoding_diffusion_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(stage: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current
    kernel sources (profiles/traffic_<stage>_<workload>.txt: 'source_sha <h>' and
    'dram_bytes_per_launch <n>' lines)."""
    path = os.path.join(ROOT, "profiles", "traffic_%s_%s.txt" % (stage, workload))
    try:
        kv = {}
        for line in open(path):
            parts = line.split()
            if len(parts) >= 2 and not line.startswith("#"):
                kv[parts[0]] = parts[1]
        if kv.get("source_sha") != source_hash():
            return None
        return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------- CPU baseline

def cpu_baseline(w, probs, seconds: float, greedy: bool = False):
    """The float64 oracle as it stands, single-threaded on a host core: sample, posterior
    (logZ and marginals of the sample) and commit, repeated for about `seconds` (greedy:
    the oracle's max-product chain)."""
    import oracle
    o = oracle.OracleFA(w.fa)
    reps, t0 = 0, time.perf_counter()
    nb = probs.shape[0]
    if greedy:
        while True:
            for b in range(nb):
                oracle.viterbi(w.fa, probs[b], w.committed[b])
            reps += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                break
        return {"value": reps * nb * w.L / el, "unit": UNIT, "cores": 1, "cpu_model": cpu_model(), "kind": "oracle",
                "sample": "%d greedy passes over %d of the %d sequences of %s (L=%d) in %.1f s, one thread"
                          % (reps, nb, w.B, w.name, w.L, el),
                "ms_per_step": 1e3 * el / reps * w.B / nb}
    if o.posterior(probs[0], w.committed[0])["empty"]:
        return {"value": None, "unit": UNIT, "cores": 1, "cpu_model": cpu_model(), "kind": "oracle",
                "sample": "none: the constrained distribution of %s at L=%d is empty" % (w.name, w.L)}
    while True:
        for b in range(nb):
            x = o.sample(probs[b], w.committed[b], 1, seed=reps)[0]
            r = o.posterior(probs[b], w.committed[b], tokens=x)
            oracle.topk(r["marg_tokens"], w.committed[b], w.k, 0, w.window)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": reps * nb * w.L / el, "unit": UNIT, "cores": 1, "cpu_model": cpu_model(), "kind": "oracle",
            "sample": "%d passes over %d of the %d sequences of %s (L=%d) in %.1f s, one thread; a whole step "
                      "of all %d sequences scales this by %d" % (reps, nb, w.B, w.name, w.L, el, w.B, w.B // nb),
            "ms_per_step": 1e3 * el / reps * w.B / nb}


def run_schedule(w, aut, stream, seed):
    """The workload's whole block-wise remasking schedule: every step is the constrained step
    and the commit, timed with CUDA events on the launching stream; the denoiser's fresh
    probabilities of each step are drawn on the device outside the events."""
    import torch
    from constrained_decoding_diffusion_gb300 import native, synth
    committed = torch.from_numpy(w.committed).cuda()
    step = native.ConstrainedStep(aut, w.B, w.L, w.k)
    n_blocks = (w.L + w.window - 1) // w.window
    per_block = max(1, w.steps // n_blocks)
    ms, i, ok = [], 0, True
    for blk in range(n_blocks):
        lo, hi = blk * w.window, min(w.L, (blk + 1) * w.window)
        for _ in range(per_block):
            probs = synth.gaussian_probs_torch(w.seed * 1000 + i, w.B, w.L, w.V, w.sigma)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                a.record(stream)
                step(probs, committed, seed, i, lo, hi, stream)
                native.fa_apply_commits(step.commit_idx, step.tokens, committed, stream)
                b.record(stream)
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b))
            ok = ok and bool((step.row_status.cpu().numpy() == 0).all())
            del probs
            i += 1
    final = committed.cpu().numpy()
    total = float(np.sum(ms))
    return {"steps": i, "blocks": n_blocks, "steps_per_block": per_block, "k": w.k, "ms_total": total,
            "ms_first_step": float(ms[0]), "ms_last_step": float(ms[-1]), "ms_mean_step": total / i,
            "value": w.B * w.L / (total / 1e3), "unit": "committed positions/s",
            "all_committed": bool((final >= 0).all()), "row_status_ok": ok,
            "timing": "per step: fa_constrained_step + fa_apply_commits between CUDA events; probabilities "
                      "drawn on the device outside them"}


def run_reference(args, rank, world):
    """The reference arm: the float64 oracle as it stands, single-threaded on a host core,
    on the same workload.  One step is a bounded sample of the workload's step: the first
    nb sequences of the batch (sample, posterior with the marginals of the sample, commit),
    nb as large as keeps one step near 20 s (the other sequences are the same computation
    on other rows); warm-up and timed steps are capped to a few minutes in all."""
    if rank != 0:
        return
    from constrained_decoding_diffusion_gb300 import synth
    import oracle
    w = synth.workload(args.workload)
    o = oracle.OracleFA(w.fa)
    probs = w.probs(n_rows=1)

    def one(seed, nb):
        for b in range(nb):
            x = o.sample(probs[b], w.committed[b], 1, seed=seed)[0]
            r = o.posterior(probs[b], w.committed[b], tokens=x)
            oracle.topk(r["marg_tokens"], w.committed[b], w.k, 0, w.window)

    t = time.perf_counter()
    one(0, 1)                    # the first warm-up step (one sequence), timed to size the run
    est1 = time.perf_counter() - t
    nb = max(1, min(w.B, int(20.0 / max(est1, 1e-6))))
    if nb > 1:
        probs = w.probs(n_rows=nb)
    est = est1 * nb
    budget = 120.0
    warm = max(1, min(args.warmup, int(0.25 * budget / max(est, 1e-6))))
    for i in range(1, warm):
        one(i, nb)
    steps = max(1, min(args.steps, int(budget / max(est, 1e-6))))
    t0 = time.perf_counter()
    for i in range(steps):
        one(i, nb)
    el = time.perf_counter() - t0
    ms = 1e3 * el / steps
    value = nb * w.L / (el / steps)
    sample = ("%d of the %d sequences of %s (L=%d) per step, %d timed steps after %d warm-up, one thread "
              "(steps capped to a %.0f s budget; a whole step of the batch takes %d times as long)"
              % (nb, w.B, w.name, w.L, steps, warm, budget, w.B // nb))
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": steps,
            "steps_requested": args.steps, "warmup": warm, "warmup_requested": args.warmup, "ms_per_step": ms,
            "ms_per_batch_step": ms * w.B / nb,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": w.name, "B": w.B, "L": w.L, "S": w.S, "V": w.V, "k": w.k,
                       "sequences_per_step": nb},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "cpu_model": cpu_model(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- native arm

def run_native(args, rank, world, local):
    import torch
    from constrained_decoding_diffusion_gb300 import native, synth

    torch.cuda.set_device(local)
    native.load()
    clocks = ClockSampler(local).__enter__()   # sampling from here on; summarised over the timed steps
    w = synth.workload(args.workload)
    if args.length is not None:
        w.L = args.length
        w.committed = np.ascontiguousarray(w.committed[:, :args.length])
        w.window = min(w.window, args.length)
    masked = int((w.committed < 0).sum())
    aut = native.fa_compile(w.fa)
    if w.B * w.L * w.V <= (1 << 27):
        probs_np = w.probs()
        probs = torch.from_numpy(probs_np).cuda()
    else:
        # large workloads: the same recipe drawn on the device; the host keeps the first
        # sequence for the CPU baseline
        probs = synth.gaussian_probs_torch(w.seed, w.B, w.L, w.V, w.sigma)
        probs_np = None
    committed = torch.from_numpy(w.committed).cuda()
    if args.method == "greedy":
        step = native.GreedyStep(aut, w.B, w.L)
        step_outputs = [step.tokens, step.score, step.row_status]
    else:
        step = native.ConstrainedStep(aut, w.B, w.L, w.k, method=args.method, confidence=args.confidence)
        step_outputs = [step.tokens, step.logZ, step.marg, step.commit_idx, step.row_status]
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    seed = 1234 + rank

    def call(offset):
        if args.method == "greedy":
            step(probs, committed)
        else:
            step(probs, committed, seed, offset, 0, w.window)

    # launches per step (counted by the library)
    with torch.cuda.stream(stream):
        n0 = native.fa_launch_count()
        call(0)
        launches_per_step = native.fa_launch_count() - n0
        for i in range(max(args.warmup, 3)):
            call(i)
    stream.synchronize()

    def capture(profiled):
        native.fa_profile_enable(profiled)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            call(0)
        native.fa_profile_enable(False)
        for _ in range(3):
            with torch.cuda.stream(stream):
                g.replay()
        stream.synchronize()
        return g

    # headline timing: a graph without the per-stage events, steps queued back to back
    graph = None if args.no_graph else capture(False)

    def run_one(i):
        if graph is not None:
            graph.replay()
        else:
            call(i)

    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks.wait_first()
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    clocks.mark_start()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush.zero_()
            ev_s[i].record(stream)
            run_one(i)
            ev_e[i].record(stream)
    torch.cuda.synchronize()
    clocks.mark_end()
    barrier(world)
    wall = time.perf_counter() - t_wall
    step_ms = [s.elapsed_time(e) for s, e in zip(ev_s, ev_e)]
    ms = float(np.mean(step_ms))
    ms_max = allreduce_max(ms, world)

    # stage attribution: a second graph carrying the library's stage events, read per step
    n_prof = min(args.steps, 200)
    stage_ms = {k: 0.0 for k in native.STAGES}
    pgraph = None if args.no_graph else capture(True)
    native.fa_profile_enable(True)
    with torch.cuda.stream(stream):
        for i in range(n_prof):
            flush.zero_()
            if pgraph is not None:
                pgraph.replay()
            else:
                call(i)
            st = native.fa_profile_read()
            for key in stage_ms:
                stage_ms[key] += st[key]
    torch.cuda.synchronize()
    native.fa_profile_enable(False)
    status = step.row_status.cpu().numpy()

    # end to end through the public call with host buffers: H2D of the step's inputs from
    # pinned memory, the step, D2H of every output, all inside the events
    h_probs = probs.cpu().pin_memory()
    h_com = torch.from_numpy(w.committed).pin_memory()
    outs = step_outputs
    h_outs = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    n_e2e = max(1, min(args.e2e_steps, args.steps))
    e2e_s = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
    e2e_e = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
    torch.cuda.synchronize()
    # the default step has a host-input entry point (fa_constrained_step_host): its copies run
    # in chunks of sequences that overlap the emission reweighting; for inputs of a few MB the
    # copies are short and a graph replay of the step after them launches faster
    use_host = args.method == "tree" and args.confidence == "marginal" and probs.numel() * 4 > (64 << 20)
    # the host-to-device copy rate of this machine for the same bytes, for context
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        c0.record(stream)
        probs.copy_(h_probs, non_blocking=True)
        c1.record(stream)
    torch.cuda.synchronize()
    h2d_gbs = probs.numel() * 4 / (c0.elapsed_time(c1) * 1e6)
    with torch.cuda.stream(stream):
        for i in range(n_e2e):
            flush.zero_()
            e2e_s[i].record(stream)
            if use_host:
                native.fa_constrained_step_host(aut, h_probs, h_com, probs, committed, seed, 0, w.k, 0, w.window,
                                                step.workspace, step.tokens, step.logZ, step.marg, step.commit_idx,
                                                step.row_status, stream)
            else:
                probs.copy_(h_probs, non_blocking=True)
                committed.copy_(h_com, non_blocking=True)
                run_one(i)
            for h, d in zip(h_outs, outs):
                h.copy_(d, non_blocking=True)
            e2e_e[i].record(stream)
    torch.cuda.synchronize()
    e2e_ms = float(np.mean([s.elapsed_time(e) for s, e in zip(e2e_s, e2e_e)]))
    e2e_ms = allreduce_max(e2e_ms, world)
    h2d = probs.numel() * 4 + committed.numel() * 4
    d2h = sum(t.numel() * t.element_size() for t in outs)

    clock_summary = clocks.summary()
    clocks.__exit__(None, None, None)
    if rank != 0:
        return
    value = replica_value(w.B * w.L, world, ms_max)
    alg = algorithmic(w, masked, args.method)
    hbm, tc, src = peaks()
    per_stage = {k: stage_ms[k] / n_prof for k in stage_ms}
    dom = max(per_stage, key=per_stage.get)
    dom_ms = per_stage[dom]
    a = alg[dom]
    achieved = a["bytes"] / (dom_ms / 1e3) / 1e9
    roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "traffic": recorded_traffic(dom, w.name),
            "algorithmic_bytes": a["bytes"], "ms": dom_ms, "peak_source": src + " (burst copy)"}
    # the whole step against its own roofline (slower of bytes at HBM peak, span FLOPs at
    # the bf16 tensor peak)
    tot_bytes = sum(v["bytes"] for v in alg.values())
    t_roof = max(tot_bytes / (hbm * 1e9), alg["upsweep"]["flops"] / (tc * 1e12))
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "L": w.L, "S": w.S, "V": w.V, "masked": masked,
                       "k": w.k, "l2": "flushed between steps (256 MiB write)",
                       "launch": "cuda_graph" if graph is not None else "eager",
                       "method": args.method, "confidence": args.confidence,
                       "parallelism": "replicas" if world > 1 else "single"},
            "roofline": roof,
            "reweight_gather": reweight_gather(w, masked, per_stage.get("reweight", 0.0), clock_summary),
            "step_roofline": {"ms_at_roofline": 1e3 * t_roof, "frac": 1e3 * t_roof / ms_max,
                              "bytes": tot_bytes, "span_flops": alg["upsweep"]["flops"]},
            "stage_ms": per_stage,
            "e2e": {"value": replica_value(w.B * w.L, world, e2e_ms), "unit": UNIT, "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "call": "fa_constrained_step_host" if use_host else "host copies + the step",
                    "h2d_copy_gbs": h2d_gbs},
            "gpu_launches": launches_per_step * args.steps, "launches_per_step": launches_per_step,
            "wall_s": wall, "row_status_ok": bool((status == 0).all()),
            "clocks": clock_summary}
    if args.schedule and w.steps > 1:
        del graph
        line["schedule"] = run_schedule(w, aut, stream, seed)
    if world == 1:
        host_probs = probs_np if probs_np is not None else probs[:1].cpu().numpy()
        line["cpu_baseline"] = cpu_baseline(w, host_probs, args.cpu_seconds, greedy=args.method == "greedy")
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_native(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
