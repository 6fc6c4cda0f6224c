#!/usr/bin/env python3
"""Benchmark: fwd+bwd of logprobs, entropy and KL (both directions) at 8192 x 75968 bf16.

One step = logprobs fwd+bwd, entropy fwd+bwd, reverse KL fwd+bwd (dA and dB)
and forward KL fwd+bwd (dA and dB) over one batch of synthetic logits of the
pages' shape (the ``pages_shape`` workload: N = 8192 rows, V = 75968, bf16,
N(0, 3^2) plus a per-row offset). ``value`` is the step's algorithmic HBM bytes
divided by its device time (GB/s); ``ms_per_step`` is the device time.

Launch: ``python bench.py [--gpus 1] [--steps K] [--warmup W] [--impl ours|reference]``;
for N > 1 under torchrun every rank runs its own 8192-row batch (rows are
independent: weak scaling, no data-path collective; one all-reduce of the
elapsed time takes the max over ranks).

``--impl reference`` times the fp64 CPU oracle on the host cores, on a bounded
sample of rows of the same workload, and reports the same metric.
"""
from __future__ import annotations

import argparse
import glob
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

METRIC = "fwd+bwd ms & HBM GB/s vs ~8 TB/s, 8192×75968 bf16 logp/entropy/KL"
UNIT = "GB/s"
N_ROWS, VOCAB = 8192, 75968
WORKLOAD = "pages' shape: 8192x75968 bf16 logits A,B ~ N(0,3^2)+U[-5,5] row offset; logprobs, entropy, " \
           "KL(A||B) and KL(B||A), each fwd+bwd (both KL gradients)"


def algorithmic_bytes(N: int, V: int, s: int = 2) -> dict:
    """HBM bytes each op must move at least once (logits and gradients; per-row vectors are < 0.01%)."""
    E = N * V * s
    return {
        "logprobs_fwd": E, "logprobs_bwd": 2 * E,
        "entropy_fwd": E, "entropy_bwd": 2 * E,
        "kl_rev_fwd": 2 * E, "kl_rev_bwd": 4 * E,
        "kl_fwd_fwd": 2 * E, "kl_fwd_bwd": 4 * E,
    }


# The step: each op's forward, then its backward, op after op. (Running the
# four forwards first and the backwards after them, in autograd order, moved
# the total by 0.3%: a kernel that follows a backward absorbs the write-back
# of its dirty L2 lines, whichever kernel that is.)
STEP_ORDER = ("logprobs_fwd", "logprobs_bwd", "entropy_fwd", "entropy_bwd",
              "kl_rev_fwd", "kl_rev_bwd", "kl_fwd_fwd", "kl_fwd_bwd")

KERNEL_OF = {  # op -> kernel name prefix in profiles (mangled names contain these)
    "logprobs_fwd": "stats_fwd_tma_kernel<0", "logprobs_bwd": "grad_kernel<0",
    "entropy_fwd": "stats_fwd_tma_kernel<1", "entropy_bwd": "grad_kernel<1",
    "kl_rev_fwd": "kl_fwd_tma_kernel", "kl_rev_bwd": "kl_grad_kernel",
    "kl_fwd_fwd": "kl_fwd_tma_kernel", "kl_fwd_bwd": "kl_grad_kernel",
}


def measured_peaks() -> dict:
    """Copy bandwidth and bf16 tensor rates (burst and sustained) measured on this machine's GPUs, else the
    fallback figures of one earlier GB300 measurement."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


def source_hash(files=None) -> str:
    """Hash of the given csrc files (all of csrc when None), to tie a recorded ncu figure to the code it measured."""
    csrc = os.path.join(ROOT, "vocab_wide_logprobs_gb300", "csrc")
    paths = sorted(glob.glob(os.path.join(csrc, "*"))) if files is None else [os.path.join(csrc, f) for f in files]
    h = hashlib.sha256()
    for f in paths:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(kernel_key: str):
    """dram read+write bytes per launch from a committed ncu summary, if it matches the current source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_key)
    if not e or e.get("source_hash") != source_hash(e.get("sources")):
        return None
    return e.get("bytes_per_launch")


def max_over_ranks(x: float, dist, device) -> float:
    """The largest of every rank's x (a job's time is its slowest rank's); x itself on one rank."""
    if not dist:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate_gbs(step_bytes: int, world: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank's step bytes over the slowest rank's step time (weak scaling)."""
    return step_bytes * world / (ms_per_step * 1e-3) / 1e9


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.tmp, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.tmp.seek(0)
        rows = [r.split(",") for r in self.tmp.read().strip().splitlines() if r.strip()]
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax = float(r[2])
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        load = [x for x in sm if smax and x > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------
def run_ours(args, rank, world, local_rank):
    import torch
    import vocab_wide_logprobs_gb300 as vp
    from vocab_wide_logprobs_gb300 import workloads

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    if args.linear_only:
        if rank == 0:
            print(json.dumps({"linear_logp": linear_bench(args, dev, N=args.linear_rows,
                                                          sustained=not args.no_sustained)}))
        if dist:
            dist.destroy_process_group()
        return

    w = workloads.pages_shape(seed=1 + rank, N=args.rows)
    a, b = w["a"].to(dev), w["b"].to(dev)
    t, g = w["targets"].to(dev), w["grad"].to(dev)
    N, V = a.shape
    nbytes = algorithmic_bytes(N, V)
    step_bytes = sum(nbytes.values())

    # outputs, allocated once (the library never allocates)
    f32 = lambda: torch.empty(N, dtype=torch.float32, device=dev)
    st = {k: f32() for k in ("lp", "H", "kl", "kl2")}
    st.update({k: vp.rowstats(N, dev) for k in ("lp_s", "H_s", "sa", "sb", "sa2", "sb2")})
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    dx = torch.empty_like(a)
    da, db = torch.empty_like(a), torch.empty_like(a)

    R, F = vp.KL_REVERSE, vp.KL_FORWARD

    def make_calls(sl, grads=None):
        """The step's eight calls on the rows `sl` of every buffer. `grads` gives each backward its own
        gradient buffers (keys of GRAD_OUTPUTS); by default the backwards share dx, da and db."""
        gr = grads or {"lp": dx, "H": dx, "ra": da, "rb": db, "fa": da, "fb": db}
        a_, b_, t_, g_ = a[sl], b[sl], t[sl], g[sl]
        d_ = {k: v[sl] for k, v in gr.items()}
        s_ = {k: v[sl] for k, v in st.items()}
        return {
            "logprobs_fwd": lambda: vp.vp_logprobs_fwd(a_, t_, 0, err, s_["lp"], s_["lp_s"]),
            "logprobs_bwd": lambda: vp.vp_logprobs_bwd(a_, t_, s_["lp_s"], g_, 0, err, d_["lp"]),
            "entropy_fwd": lambda: vp.vp_entropy_fwd(a_, s_["H"], s_["H_s"]),
            "entropy_bwd": lambda: vp.vp_entropy_bwd(a_, s_["H_s"], g_, d_["H"]),
            "kl_rev_fwd": lambda: vp.vp_kl_fwd(a_, b_, R, s_["kl"], s_["sa"], s_["sb"]),
            "kl_rev_bwd": lambda: vp.vp_kl_bwd(a_, b_, R, s_["sa"], s_["sb"], g_, da=d_["ra"], db=d_["rb"]),
            "kl_fwd_fwd": lambda: vp.vp_kl_fwd(a_, b_, F, s_["kl2"], s_["sa2"], s_["sb2"]),
            "kl_fwd_bwd": lambda: vp.vp_kl_bwd(a_, b_, F, s_["sa2"], s_["sb2"], g_, da=d_["fa"], db=d_["fb"]),
        }

    calls = make_calls(slice(None))

    def op(name):
        calls[name]()

    ops = list(STEP_ORDER)
    launches_per_step = len(ops)

    def step(events=None):
        for i, name in enumerate(ops):
            if events is not None:
                events[i][0].record()
            op(name)
            if events is not None:
                events[i][1].record()

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()

    # The timed region holds the steps' kernels back to back, with no event between them (an event
    # between two kernels would also stop the next one from being scheduled while the previous one
    # finishes); the per-op breakdown comes from a second pass of the same steps with an event pair
    # around every call.
    stream = torch.cuda.current_stream()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for k in range(args.steps):
            step()
        stop.record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
    elapsed_ms = max_over_ranks(start.elapsed_time(stop), dist, dev)
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in ops]
          for _ in range(args.steps)]
    for k in range(args.steps):
        step(ev[k])
    torch.cuda.synchronize()
    per_op_ms = {name: statistics.median(ev[k][i][0].elapsed_time(ev[k][i][1]) for k in range(args.steps))
                 for i, name in enumerate(ops)}
    ms_per_step = elapsed_ms / args.steps
    value = job_rate_gbs(step_bytes, world, ms_per_step)

    # dominant kernel (largest share of the step) and its roofline
    dom = max(per_op_ms, key=per_op_ms.get)
    peaks = measured_peaks()
    achieved = nbytes[dom] / (per_op_ms[dom] * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": KERNEL_OF[dom], "op": dom, "achieved": round(achieved, 1),
                "peak": peaks["hbm_gbs"], "peak_src": peaks["src"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic_for(dom),
                "algorithmic_bytes": nbytes[dom]}

    # the end-to-end step right after the device-timed one, before the other workloads
    e2e = None
    if not args.no_e2e:
        per_row = end_to_end(args, w, a, b, t, g, st, ops, make_calls, step_bytes, world, dist, stream, dev,
                             with_grads=False)
        e2e = end_to_end(args, w, a, b, t, g, st, ops, make_calls, step_bytes, world, dist, stream, dev,
                         with_grads=True)
        e2e["per_row_outputs_only"] = per_row

    table = ops_table(per_op_ms, nbytes, peaks, kl_da_only_ms(a, b, g, dev)) if rank == 0 else None
    jsd = jsd_bench(args, a, b, g, dev, peaks) if rank == 0 else None
    topk = topk_bench(args, a, dev, peaks) if rank == 0 else None
    strided = strided_bench(args, dev, peaks, st, err, dx, da, db) if rank == 0 and not args.no_strided else None
    stress = stress_bench(args, dev, peaks) if rank == 0 and not args.no_strided else None
    short = short_batch_bench(args, dev, peaks) if rank == 0 and not args.no_strided else None

    linear = None
    if not args.no_linear and rank == 0:
        with ClockSampler(local_rank) as lin_clocks:
            linear = linear_bench(args, dev, N=args.linear_rows, sustained=not args.no_sustained)
        linear["clocks"] = lin_clocks.summary()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, seconds=args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "N": N, "V": V, "rows_per_gpu": N, "parallelism": f"dp{world}",
                       "order": "each op's forward, then its backward",
                       "l2": "inputs larger than L2 (1.245 GB per logits tensor)",
                       "algorithmic_bytes_per_step": step_bytes},
            "per_op_ms": {k: round(v, 4) for k, v in per_op_ms.items()},
            "per_op_gbs": {k: round(nbytes[k] / (v * 1e-3) / 1e9, 1) for k, v in per_op_ms.items()},
            "ops_table": table,
            "roofline": roofline, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks.summary(), "cpu_baseline": cpu, "jsd": jsd, "topk": topk, "strided": strided, "fp32_stress": stress,
            "short_batch": short, "linear_logp": linear,
        }
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


def jsd_bench(args, a, b, g, dev, peaks, beta=0.5):
    """Generalized JSD (interior beta) on the step's buffers: two-pass forward and both gradients."""
    import torch
    import vocab_wide_logprobs_gb300 as vp
    N, V = a.shape
    E2 = 2 * N * V * a.element_size()           # one read of A and B
    jsd, sa, sb = vp.vp_jsd_fwd(a, b, beta)
    da, db = torch.empty_like(a), torch.empty_like(a)
    fwd = lambda: vp.vp_jsd_fwd(a, b, beta, jsd=jsd, stats_a=sa, stats_b=sb)
    bwd = lambda: vp.vp_jsd_bwd(a, b, beta, sa, sb, g, da=da, db=db)
    for _ in range(3):
        fwd()
        bwd()
    torch.cuda.synchronize()
    reps = max(3, min(args.steps, 10))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    tf = tb = 0.0
    for _ in range(reps):
        ev[0].record()
        fwd()
        ev[1].record()
        bwd()
        ev[2].record()
        torch.cuda.synchronize()
        tf += ev[0].elapsed_time(ev[1])
        tb += ev[1].elapsed_time(ev[2])
    tf, tb = tf / reps, tb / reps
    gbs = lambda nbytes, ms: round(nbytes / (ms * 1e-3) / 1e9, 1)
    return {"workload": f"{N}x{V} bf16, beta={beta}, gradients to both inputs", "fwd_ms": round(tf, 4),
            "bwd_ms": round(tb, 4), "fwd_gbs": gbs(2 * E2, tf), "bwd_gbs": gbs(2 * E2, tb),
            "fwd_bytes": 2 * E2, "bwd_bytes": 2 * E2,
            "note": "forward = two reads of A and B (statistics, then both KL-to-mixture sums); "
                    "backward = one read of A and B and one write of dA and dB",
            "frac_of_copy_peak": {"fwd": round(2 * E2 / (tf * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                                  "bwd": round(2 * E2 / (tb * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}}


def strided_bench(args, dev, peaks, st, err, dx, da, db):
    """The step's eight calls on the strided workload: x[:, :-1] of [B, 513, 75968] bf16 tensors (512 rows
    per outer index addressed with two strides, read in place; B = ceil(rows / 512), 16 at the default 8192
    rows), into the step's contiguous outputs, or into its own where its row count differs from the step's."""
    import torch
    import vocab_wide_logprobs_gb300 as vp
    from vocab_wide_logprobs_gb300 import workloads
    w = workloads.strided(B=max(1, -(-args.rows // 512)))
    af, bf = w["a_full"].to(dev), w["b_full"].to(dev)
    t, g = w["targets"].reshape(-1).to(dev), w["grad"].reshape(-1).to(dev)
    del w
    a, b = af[:, :-1], bf[:, :-1]
    N, V = a.shape[0] * a.shape[1], a.shape[2]
    if dx.shape != (N, V):   # the step's outputs hold another number of rows
        f32 = lambda: torch.empty(N, dtype=torch.float32, device=dev)
        st = {k: f32() for k in ("lp", "H", "kl", "kl2")}
        st.update({k: vp.rowstats(N, dev) for k in ("lp_s", "H_s", "sa", "sb", "sa2", "sb2")})
        dx, da, db = (torch.empty((N, V), dtype=a.dtype, device=dev) for _ in range(3))
    R, F = vp.KL_REVERSE, vp.KL_FORWARD
    calls = {
        "logprobs_fwd": lambda: vp.vp_logprobs_fwd(a, t, 0, err, st["lp"], st["lp_s"]),
        "logprobs_bwd": lambda: vp.vp_logprobs_bwd(a, t, st["lp_s"], g, 0, err, dx),
        "entropy_fwd": lambda: vp.vp_entropy_fwd(a, st["H"], st["H_s"]),
        "entropy_bwd": lambda: vp.vp_entropy_bwd(a, st["H_s"], g, dx),
        "kl_rev_fwd": lambda: vp.vp_kl_fwd(a, b, R, st["kl"], st["sa"], st["sb"]),
        "kl_rev_bwd": lambda: vp.vp_kl_bwd(a, b, R, st["sa"], st["sb"], g, da=da, db=db),
        "kl_fwd_fwd": lambda: vp.vp_kl_fwd(a, b, F, st["kl2"], st["sa2"], st["sb2"]),
        "kl_fwd_bwd": lambda: vp.vp_kl_bwd(a, b, F, st["sa2"], st["sb2"], g, da=da, db=db),
    }
    line = _time_calls(args, calls, STEP_ORDER, algorithmic_bytes(N, V), peaks)
    del af, bf
    return {"workload": f"x[:, :-1] of [{a.shape[0]}, 513, {V}] bf16 tensors A and B: {N} rows, 512 per outer "
                        "index, read in place with two row strides; gradients written contiguous", **line}


def _time_calls(args, calls, order, nbytes, peaks):
    """Per-call CUDA-event times of `calls` run in `order` (3 untimed rounds, then the mean of several), as
    the step's ms, GB/s over the algorithmic bytes `nbytes` and per-call GB/s."""
    import torch
    for _ in range(3):
        for name in order:
            calls[name]()
    torch.cuda.synchronize()
    reps = max(3, min(args.steps, 10))
    ev = {k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for k in order}
    per_op = {k: 0.0 for k in order}
    for _ in range(reps):
        for name in order:
            ev[name][0].record()
            calls[name]()
            ev[name][1].record()
        torch.cuda.synchronize()
        for name in order:
            per_op[name] += ev[name][0].elapsed_time(ev[name][1]) / reps
    ms = sum(per_op.values())
    total = sum(nbytes[k] for k in order)
    return {"ms_per_step": round(ms, 4), "value_gbs": round(total / (ms * 1e-3) / 1e9, 1),
            "frac_of_copy_peak": round(total / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "per_op_gbs": {k: round(nbytes[k] / (v * 1e-3) / 1e9, 1) for k, v in per_op.items()}}


NOMINAL_HBM_GBS = 8000.0   # the pages' "about 8 TB/s"


def ops_table(per_op_ms, nbytes, peaks, kl_da_only_ms):
    """Each op's fwd + bwd (in-step medians) against the nominal 8 TB/s and the measured copy peak, with
    the 85%-of-8-TB/s mark; KL with dA only (the pages' timing model) from its own timed calls."""
    rows = {"logprobs": ("logprobs_fwd", "logprobs_bwd"), "entropy": ("entropy_fwd", "entropy_bwd"),
            "kl_da_db": ("kl_rev_fwd", "kl_rev_bwd")}
    out = {}
    for name, (f, b) in rows.items():
        ms = per_op_ms[f] + per_op_ms[b]
        out[name] = (ms, nbytes[f] + nbytes[b])
    E2 = nbytes["logprobs_fwd"]                      # E * s
    out["kl_da_only"] = (kl_da_only_ms, 5 * E2)      # read A, B twice, write dA
    table = {}
    for name, (ms, by) in out.items():
        gbs = by / (ms * 1e-3) / 1e9
        table[name] = {"ms": round(ms, 4), "bytes": by, "gbs": round(gbs, 1),
                       "frac_of_8tbps": round(gbs / NOMINAL_HBM_GBS, 4),
                       "frac_of_measured_copy": round(gbs / peaks["hbm_gbs"], 4),
                       "mark_85pct_of_8tbps_ms": round(by / (0.85 * NOMINAL_HBM_GBS * 1e9) * 1e3, 4)}
    return table


def kl_da_only_ms(a, b, g, dev, reps=20):
    """KL(A||B) forward plus the backward with dA only (a detached teacher), median of `reps` back-to-back
    pairs after 5 warm-ups, CUDA events on the launching stream."""
    import torch
    import vocab_wide_logprobs_gb300 as vp
    N = a.shape[0]
    kl = torch.empty(N, dtype=torch.float32, device=dev)
    sa, sb = vp.rowstats(N, dev), vp.rowstats(N, dev)
    da = torch.empty_like(a)

    def pair():
        vp.vp_kl_fwd(a, b, vp.KL_REVERSE, kl, sa, sb)
        vp.vp_kl_bwd(a, b, vp.KL_REVERSE, sa, sb, g, want_db=False, da=da)

    for _ in range(5):
        pair()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for e0, e1 in ev:
        e0.record()
        pair()
        e1.record()
    torch.cuda.synchronize()
    return statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)


def short_batch_bench(args, dev, peaks, rows=1024, reps=10):
    """The step's eight calls on a short batch (1024 rows of the pages' shape, 155.6 MB per logits tensor,
    near the 129 MB L2), under both row-split settings of the forward scans. Before every timed call the
    L2 is flushed: a 256 MiB buffer is written, then another 256 MiB buffer is read, so that the call
    neither finds its inputs in L2 nor pays for the write-back of the flush's dirty lines. Calls are
    queued back to back (no host synchronisation until the end), so the host's launch latency is not
    counted either; each call is bracketed by CUDA events on the launching stream."""
    import torch
    import vocab_wide_logprobs_gb300 as vp
    from vocab_wide_logprobs_gb300 import workloads
    w = workloads.pages_shape(seed=7, N=rows)
    a, b, t, g = (w[k].to(dev) for k in ("a", "b", "targets", "grad"))
    N, V = a.shape
    nbytes = algorithmic_bytes(N, V)
    R, F = vp.KL_REVERSE, vp.KL_FORWARD
    f32 = lambda: torch.empty(N, dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    o = {k: f32() for k in ("lp", "H", "kl", "kl2")}
    s = {k: vp.rowstats(N, dev) for k in ("lp", "H", "a", "b", "a2", "b2")}
    dx, da, db = torch.empty_like(a), torch.empty_like(a), torch.empty_like(a)
    calls = {
        "logprobs_fwd": lambda: vp.vp_logprobs_fwd(a, t, 0, err, o["lp"], s["lp"]),
        "logprobs_bwd": lambda: vp.vp_logprobs_bwd(a, t, s["lp"], g, 0, err, dx),
        "entropy_fwd": lambda: vp.vp_entropy_fwd(a, o["H"], s["H"]),
        "entropy_bwd": lambda: vp.vp_entropy_bwd(a, s["H"], g, dx),
        "kl_rev_fwd": lambda: vp.vp_kl_fwd(a, b, R, o["kl"], s["a"], s["b"]),
        "kl_rev_bwd": lambda: vp.vp_kl_bwd(a, b, R, s["a"], s["b"], g, da=da, db=db),
        "kl_fwd_fwd": lambda: vp.vp_kl_fwd(a, b, F, o["kl2"], s["a2"], s["b2"]),
        "kl_fwd_bwd": lambda: vp.vp_kl_bwd(a, b, F, s["a2"], s["b2"], g, da=da, db=db),
    }
    dirty = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    clean = torch.zeros(256 << 20, dtype=torch.uint8, device=dev)

    def flush():
        dirty.fill_(1)
        clean.sum()

    out = {"workload": f"pages shape, N={N}, V={V}, bf16", "reps": reps,
           "l2": "flushed before every call: 256 MiB written, then 256 MiB read", "launch": "queued back to back"}
    old = vp.vp_get_row_split()
    try:
        for split in (1, 2):
            vp.vp_set_row_split(split)
            for _ in range(3):
                for name in STEP_ORDER:
                    flush()
                    calls[name]()
            torch.cuda.synchronize()
            ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in STEP_ORDER]
                  for _ in range(reps)]
            for k in range(reps):
                for i, name in enumerate(STEP_ORDER):
                    flush()
                    ev[k][i][0].record()
                    calls[name]()
                    ev[k][i][1].record()
            torch.cuda.synchronize()
            per_op = {name: statistics.mean(ev[k][i][0].elapsed_time(ev[k][i][1]) for k in range(reps))
                      for i, name in enumerate(STEP_ORDER)}
            ms = sum(per_op.values())
            total = sum(nbytes.values())
            out[f"row_split_{split}"] = {
                "ms_per_step": round(ms, 4), "value_gbs": round(total / (ms * 1e-3) / 1e9, 1),
                "frac_of_copy_peak": round(total / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                "per_op_us": {k: round(v * 1e3, 1) for k, v in per_op.items()},
                "per_op_gbs": {k: round(nbytes[k] / (v * 1e-3) / 1e9, 1) for k, v in per_op.items()}}
    finally:
        vp.vp_set_row_split(old)
    out["default"] = f"row_split_{old}"
    return out


def stress_bench(args, dev, peaks):
    """The fp32 numerics-stress workload: entropy and KL in both directions, fwd and bwd (gradients to
    both inputs), on [N, 75968] fp32 rows (N = --rows, 8192 by default) offset by 1e4 with 1% of B masked
    to -inf, so that KL(A||B) is +inf on essentially every row and KL(B||A) runs the zero-weight path at a
    large offset."""
    import torch
    import vocab_wide_logprobs_gb300 as vp
    from vocab_wide_logprobs_gb300 import workloads
    w = workloads.numerics_stress(N=args.rows)
    a, b, g = w["a"].to(dev), w["b"].to(dev), w["grad"].to(dev)
    del w
    N, V = a.shape
    f32 = lambda: torch.empty(N, dtype=torch.float32, device=dev)
    o = {k: f32() for k in ("H", "kl", "kl2")}
    o.update({k: vp.rowstats(N, dev) for k in ("H_s", "sa", "sb", "sa2", "sb2")})
    dx, da, db = torch.empty_like(a), torch.empty_like(a), torch.empty_like(a)
    R, F = vp.KL_REVERSE, vp.KL_FORWARD
    calls = {
        "entropy_fwd": lambda: vp.vp_entropy_fwd(a, o["H"], o["H_s"]),
        "entropy_bwd": lambda: vp.vp_entropy_bwd(a, o["H_s"], g, dx),
        "kl_rev_fwd": lambda: vp.vp_kl_fwd(a, b, R, o["kl"], o["sa"], o["sb"]),
        "kl_rev_bwd": lambda: vp.vp_kl_bwd(a, b, R, o["sa"], o["sb"], g, da=da, db=db),
        "kl_fwd_fwd": lambda: vp.vp_kl_fwd(a, b, F, o["kl2"], o["sa2"], o["sb2"]),
        "kl_fwd_bwd": lambda: vp.vp_kl_bwd(a, b, F, o["sa2"], o["sb2"], g, da=da, db=db),
    }
    order = [k for k in STEP_ORDER if k in calls]
    line = _time_calls(args, calls, order, algorithmic_bytes(N, V, s=4), peaks)
    del a, b, dx, da, db
    return {"workload": f"{N}x{V} fp32, N(0, 9) + 1e4 on every row of A and B, 1% of B set to -inf; entropy "
                        "and KL both directions, fwd+bwd", **line}


def topk_bench(args, a, dev, peaks, K=20):
    """Logprobs of K ids per row (top-k) on the step's logits A: one scan forward, one read + one write backward."""
    import torch
    import vocab_wide_logprobs_gb300 as vp
    from vocab_wide_logprobs_gb300 import workloads
    N, V = a.shape
    ids = workloads.topk_ids(seed=101, N=N, V=V, K=K)
    t, g = ids["targets"].to(dev), ids["grad"].to(dev)
    lp, st = vp.vp_logprobs_topk_fwd(a, t)
    dx = torch.empty_like(a)
    reps = max(3, min(args.steps, 10))
    tf = _time_ms(lambda: vp.vp_logprobs_topk_fwd(a, t, logp=lp, stats=st), reps)
    tb = _time_ms(lambda: vp.vp_logprobs_topk_bwd(a, t, st, g, dx=dx), reps)
    E = N * V * a.element_size()
    fb, bb = E + 16 * N * K, 2 * E + 12 * N * K
    gbs = lambda nbytes, ms: round(nbytes / (ms * 1e-3) / 1e9, 1)
    return {"workload": f"{N}x{V} bf16, K={K} ids per row (10% duplicates, 10% ignored)", "fwd_ms": round(tf, 4),
            "bwd_ms": round(tb, 4), "fwd_gbs": gbs(fb, tf), "bwd_gbs": gbs(bb, tb), "fwd_bytes": fb,
            "bwd_bytes": bb, "frac_of_copy_peak": {"fwd": round(fb / (tf * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                                                   "bwd": round(bb / (tb * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}}


def _time_ms(fn, reps, idle_s=0.0):
    """Mean ms of fn over reps calls, CUDA events on the current stream, after one untimed call
    (and idle_s seconds of idle GPU, so that a burst is timed from the same power state)."""
    import torch
    fn()
    torch.cuda.synchronize()
    if idle_s > 0:
        time.sleep(idle_s)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


IDLE_S = 1.0   # idle seconds before each timed burst of the linear ops
SUSTAINED_CALLS = 20   # back-to-back calls of each linear op in the sustained figures


def linear_bench(args, dev, N=8192, V=75968, D=4096, sustained=True):
    """Fused linear ops on the linear workload (hidden [8192, 4096], W [75968, 4096] bf16): logp, entropy,
    KL against a second model of the same shape and the generalized JSD, forward and backward, the
    backwards at both precisions (exact: dz as a bf16 pair, the default; fast: dz rounded to bf16).
    Each op is timed as a burst of three calls after IDLE_S seconds of idle GPU, against the measured
    burst bf16 peak; with `sustained`, also as SUSTAINED_CALLS back-to-back calls, against the measured
    sustained peak (a training step runs these GEMMs back to back under the power cap)."""
    import torch
    import vocab_wide_logprobs_gb300 as vp
    from vocab_wide_logprobs_gb300 import workloads
    w = workloads.linear(N=N, V=V, D=D)
    h, W, t = w["hidden"].to(dev), w["weight"].to(dev), w["targets"].to(dev)
    g = w["grad"].to(dev)
    logp = torch.empty(N, dtype=torch.float32, device=dev)
    st = vp.rowstats(N, dev)
    peaks = measured_peaks()
    burst_peak, sus_peak = peaks.get("bf16_tflops"), peaks.get("bf16_tflops_sustained")
    unit = 2.0 * N * V * D          # one GEMM of the logits' shape
    EXACT, FAST = vp.GRAD_EXACT, vp.GRAD_FAST
    reps = 3   # a burst of three calls

    ws = torch.empty(vp.vp_linear_logp_workspace_size(N, V, D), dtype=torch.uint8, device=dev)
    dh, dW = torch.empty_like(h), torch.empty_like(W)
    wsb = torch.empty(vp.vp_linear_logp_bwd_workspace_size(N, V, D), dtype=torch.uint8, device=dev)
    H = torch.empty(N, dtype=torch.float32, device=dev)
    wse = torch.empty(max(vp._lib.lib().vp_linear_entropy_bwd_workspace_size(N, V, D),
                          vp._lib.lib().vp_linear_entropy_workspace_size(N, V, D)), dtype=torch.uint8, device=dev)
    tw = workloads.linear(seed=14, N=N, V=V, D=D)
    hb, Wb = tw["hidden"].to(dev), tw["weight"].to(dev)
    del tw
    kl = torch.empty(N, dtype=torch.float32, device=dev)
    sb = vp.rowstats(N, dev)
    wsk = torch.empty(vp._lib.lib().vp_linear_kl_bwd_workspace_size(N, V, D, D), dtype=torch.uint8, device=dev)
    outs = [dh, dW, torch.empty_like(hb), torch.empty_like(Wb)]
    R = vp.KL_REVERSE
    # (name, call, GEMM units of 2 N V D flops)
    ops = [
        ("logp_fwd", lambda: vp.vp_linear_logp_fwd(h, W, t, logp=logp, stats=st, workspace=ws), 1),
        ("logp_bwd", lambda: vp.vp_linear_logp_bwd(h, W, t, st, g, dhidden=dh, dW=dW, workspace=wsb), 5),
        ("logp_bwd_fast", lambda: vp.vp_linear_logp_bwd(h, W, t, st, g, dhidden=dh, dW=dW, workspace=wsb,
                                                        precision=FAST), 3),
        ("entropy_fwd", lambda: vp.vp_linear_entropy_fwd(h, W, H=H, stats=st, workspace=wse), 1),
        ("entropy_bwd", lambda: vp.vp_linear_entropy_bwd(h, W, st, g, dhidden=dh, dW=dW, workspace=wse), 5),
        ("entropy_bwd_fast", lambda: vp.vp_linear_entropy_bwd(h, W, st, g, dhidden=dh, dW=dW, workspace=wse,
                                                              precision=FAST), 3),
        ("kl_fwd", lambda: vp.vp_linear_kl_fwd(h, W, hb, Wb, R, kl=kl, stats_a=st, stats_b=sb, workspace=wsk), 2),
        ("kl_bwd", lambda: vp.vp_linear_kl_bwd(h, W, hb, Wb, R, st, sb, g, outs=outs, workspace=wsk), 10),
        ("kl_bwd_fast", lambda: vp.vp_linear_kl_bwd(h, W, hb, Wb, R, st, sb, g, outs=outs, workspace=wsk,
                                                    precision=FAST), 6),
        ("jsd_fwd", lambda: vp.vp_linear_jsd_fwd(h, W, hb, Wb, 0.5, jsd=kl, stats_a=st, stats_b=sb, workspace=wsk),
         4),
        ("jsd_bwd", lambda: vp.vp_linear_jsd_bwd(h, W, hb, Wb, 0.5, st, sb, g, outs=outs, workspace=wsk), 10),
        ("jsd_bwd_fast", lambda: vp.vp_linear_jsd_bwd(h, W, hb, Wb, 0.5, st, sb, g, outs=outs, workspace=wsk,
                                                      precision=FAST), 6),
    ]
    # the records each backward reads: the matching forward runs right before it
    fwd_of = {"logp": 0, "entropy": 3, "kl": 6, "jsd": 9}
    families = getattr(args, "linear_ops", None)
    if families:   # a subset of the op families (a small profiling run)
        keep = set(families.split(",")) & set(fwd_of)
        ops = [o for o in ops if o[0].split("_")[0] in keep]
        fwd_of = {f: next(j for j, o in enumerate(ops) if o[0] == f + "_fwd") for f in keep}
    burst, sus = {}, {}
    for k, (name, fn, units) in enumerate(ops):
        if not name.endswith("_fwd"):
            ops[fwd_of[name.split("_")[0]]][1]()
        ms = _time_ms(fn, reps, IDLE_S)
        burst[name] = (ms, units * unit / (ms * 1e-3) / 1e12)
    clocks = None
    if sustained:
        with ClockSampler(dev.index or 0) as ck:
            for name, fn, units in ops:
                if name.endswith("_fast"):
                    continue
                if not name.endswith("_fwd"):
                    ops[fwd_of[name.split("_")[0]]][1]()
                ms = _time_ms(fn, SUSTAINED_CALLS)
                sus[name] = (ms, units * unit / (ms * 1e-3) / 1e12)
        clocks = ck.summary()
    del ws, wsb, wse, wsk, outs, hb, Wb
    torch.cuda.empty_cache()

    frac = lambda x, pk: round(x / pk, 4) if pk else None

    def entry(op, fwd_units, bwd_units, fast_units, what):
        f, b, bf = burst[op + "_fwd"], burst[op + "_bwd"], burst[op + "_bwd_fast"]
        e = {"workload": what, "fwd_ms": round(f[0], 4), "bwd_ms": round(b[0], 4), "bwd_fast_ms": round(bf[0], 4),
             "fwd_tflops": round(f[1], 1), "bwd_tflops": round(b[1], 1), "bwd_fast_tflops": round(bf[1], 1),
             "fwd_frac": frac(f[1], burst_peak), "bwd_frac": frac(b[1], burst_peak),
             "bwd_fast_frac": frac(bf[1], burst_peak),
             "flops": {"fwd": fwd_units * unit, "bwd": bwd_units * unit, "bwd_fast": fast_units * unit}}
        if sus:
            sf, sbw = sus[op + "_fwd"], sus[op + "_bwd"]
            e["sustained"] = {"calls": SUSTAINED_CALLS, "fwd_ms": round(sf[0], 4), "bwd_ms": round(sbw[0], 4),
                              "fwd_tflops": round(sf[1], 1), "bwd_tflops": round(sbw[1], 1),
                              "fwd_frac": frac(sf[1], sus_peak), "bwd_frac": frac(sbw[1], sus_peak),
                              "peak": sus_peak, "peak_src": "measured bf16 sustained"}
        return e

    have = {name.split("_")[0] for name, _, _ in ops}
    out = {}
    if "logp" in have:
        out = entry("logp", 1, 5, 3, f"hidden [{N},{D}] x W [{V},{D}] bf16, logp of uniform targets")
        out["roofline"] = {"bound": "tensor", "achieved": out["fwd_tflops"], "peak": burst_peak, "unit": "TFLOP/s",
                           "peak_src": "measured bf16 burst" if burst_peak else None, "frac": out["fwd_frac"],
                           "flops": unit}
        out["bwd_roofline"] = {"bound": "tensor", "achieved": out["bwd_tflops"], "peak": burst_peak,
                               "unit": "TFLOP/s", "frac": out["bwd_frac"], "flops": 5 * unit,
                               "note": "exact precision: logits recomputed (2NVD), dhidden and dW with dz_hi and "
                                       "dz_lo (4NVD each); fast precision: 3 GEMMs of 2NVD"}
    if "entropy" in have:
        out["entropy"] = entry("entropy", 1, 5, 3, "entropy of softmax(h W^T); backward: logits, dhidden, dW")
    if "kl" in have:
        out["kl"] = entry("kl", 2, 10, 6, "KL(A||B) of two models of this shape; forward: both logits tiles; "
                          "backward: both logits tiles, dhidden and dW of both models")
    if "jsd" in have:
        out["jsd"] = entry("jsd", 4, 10, 6, "generalized JSD (beta = 0.5) of the two models; forward: two passes "
                           "of both logits tiles; backward: as for KL")
    out["sustained_clocks"] = clocks
    return out


GRAD_OUTPUTS = ("lp", "H", "ra", "rb", "fa", "fb")   # dlogits of logprobs, entropy; dA, dB of both KLs


def end_to_end(args, w, a, b, t, g, st, ops, make_calls, step_bytes, world, dist, stream, dev, chunks=8,
               with_grads=True):
    """The step end to end through the public API with host buffers.

    Every step copies the step's inputs from pinned host memory, runs the eight
    calls and copies the step's results back to pinned host memory: the four
    per-row outputs and, with `with_grads`, all six gradients the step produces
    (each backward then writes its own gradient buffer). Rows are independent,
    so the step is cut into `chunks` row blocks: block k's host-to-device copy
    runs on an upload stream and block k - 1's results go back on a download
    stream while the calls of the blocks between run on the compute stream."""
    import torch
    import vocab_wide_logprobs_gb300 as vp
    N = a.shape[0]
    # pinned host buffers on the GPU's own NUMA node (first touch under a CPU
    # affinity local to the GPU); a buffer on the far node halves the copy rate
    numa = _gpu_local_cpus(dev)
    saved = os.sched_getaffinity(0) if numa else None
    if numa:
        os.sched_setaffinity(0, numa)
    try:
        h_a, h_b = w["a"].pin_memory(), w["b"].pin_memory()
        h_t, h_g = w["targets"].pin_memory(), w["grad"].pin_memory()
        h_out = torch.empty(4, N, dtype=torch.float32).pin_memory()
        h_grads = ({k: torch.empty(a.shape, dtype=a.dtype, pin_memory=True) for k in GRAD_OUTPUTS}
                   if with_grads else {})
    finally:
        if saved:
            os.sched_setaffinity(0, saved)
    grads = {k: torch.empty_like(a) for k in GRAD_OUTPUTS} if with_grads else None
    h2d = sum(x.numel() * x.element_size() for x in (h_a, h_b, h_t, h_g))
    d2h = h_out.numel() * 4 + sum(x.numel() * x.element_size() for x in h_grads.values())
    chunks = max(1, min(chunks, N))
    bounds = [N * k // chunks for k in range(chunks + 1)]
    blocks = [slice(bounds[k], bounds[k + 1]) for k in range(chunks)]
    calls = [make_calls(sl, grads) for sl in blocks]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    landed = [torch.cuda.Event() for _ in blocks]   # block k's inputs are on the device
    read = [torch.cuda.Event() for _ in blocks]     # block k's calls are done (inputs read, results written)
    fetched = [torch.cuda.Event() for _ in blocks]  # block k's results are in host memory

    # each block's host and device views, made once (the step then only issues calls)
    ups = [[(dst[sl], src[sl]) for dst, src in ((a, h_a), (b, h_b), (t, h_t), (g, h_g))] for sl in blocks]
    downs = [[(h_out[i, sl], st[key][sl]) for i, key in enumerate(("lp", "H", "kl", "kl2"))]
             + [(h_grads[k][sl], grads[k][sl]) for k in h_grads] for sl in blocks]

    def e2e_step():
        for k in range(len(blocks)):
            with torch.cuda.stream(up):
                up.wait_event(read[k])              # the previous step is done with these rows
                for dst, src in ups[k]:
                    vp.vp_upload(dst, src)
                landed[k].record(up)
            stream.wait_event(landed[k])
            stream.wait_event(fetched[k])           # the previous step's results of these rows are out
            for name in ops:
                calls[k][name]()
            read[k].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(read[k])
                for dst, src in downs[k]:
                    vp.vp_download(dst, src)
                fetched[k].record(down)

    e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    a.copy_(h_a, non_blocking=True)                 # the host link alone, for the record
    e1.record(stream)
    torch.cuda.synchronize()
    h2d_gbs = a.numel() * a.element_size() / (e0.elapsed_time(e1) * 1e-3) / 1e9
    e2e_steps = max(3, min(args.steps, 10))
    e0.record(stream)
    up.wait_event(e0)
    h0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    enqueue_ms = (time.perf_counter() - h0) * 1e3 / e2e_steps   # host time to issue one step's calls
    for ev in fetched:
        stream.wait_event(ev)                       # the timed region ends when the last results are out
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dist, dev)
    out = {"value": round(job_rate_gbs(step_bytes, world, e2e_ms), 1), "unit": UNIT,
           "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "results_copied_back": ("per-row outputs and all six gradients (dlogits of logprobs and entropy, "
                                   "dA and dB of both KL directions)") if with_grads else "per-row outputs only",
           "pipeline": f"{chunks} row blocks; uploads (vp_upload) and downloads (vp_download) on their own "
                       "streams overlap the calls",
           "h2d_link_gbs": round(h2d_gbs, 1), "host_buffers_numa_local": bool(numa),
           "host_enqueue_ms_per_step": round(enqueue_ms, 3)}
    del grads, h_grads
    return out


def _gpu_local_cpus(dev):
    """CPUs local to the GPU's NUMA node (sysfs), or None when that cannot be read."""
    import torch
    try:
        p = torch.cuda.get_device_properties(dev)
        bus = f"{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        with open(f"/sys/bus/pci/devices/{bus}/local_cpulist") as f:
            spec = f.read().strip()
        cpus = set()
        for part in spec.split(","):
            lo, _, hi = part.partition("-")
            cpus.update(range(int(lo), int(hi or lo) + 1))
        cpus &= os.sched_getaffinity(0)
        return cpus or None
    except (AttributeError, OSError, ValueError):
        return None


# ---------------------------------------------------------------------------
# the oracle on the host cores
# ---------------------------------------------------------------------------
def _oracle_rows(w, rows):
    import numpy as np
    import oracle
    a64 = w["a"][rows].double().numpy()
    b64 = w["b"][rows].double().numpy()
    t = w["targets"][rows].numpy()
    g = w["grad"][rows].double().numpy()

    def run():
        lp = oracle.logprobs_fwd(a64, t)
        oracle.logprobs_bwd(a64, t, g)
        oracle.entropy_fwd(a64)
        oracle.entropy_bwd(a64, g)
        for d in (oracle.REVERSE, oracle.FORWARD):
            oracle.kl_fwd(a64, b64, d)
            oracle.kl_bwd(a64, b64, g, d)
        return lp
    return run, np


def _oracle_rate(run, batch_rows, seconds):
    """GB/s of the oracle running `run` (batch_rows rows per call) until `seconds` pass; (rate, rows, s)."""
    t0 = time.perf_counter()
    reps = 0
    while True:
        run()
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    rows = reps * batch_rows
    return sum(algorithmic_bytes(rows, VOCAB).values()) / dt / 1e9, rows, dt


def cpu_baseline(w, seconds=12.0, batch_rows=64, single_seconds=4.0):
    """The oracle as it stands, all four ops fwd+bwd, on batches of rows until `seconds` pass, with
    OpenMP over rows on all host cores; then on one thread for `single_seconds` (8 rows per call)."""
    import oracle
    run, _ = _oracle_rows(w, slice(0, batch_rows))
    cores = oracle.num_threads()
    rate, rows, dt = _oracle_rate(run, batch_rows, seconds)
    run1, _ = _oracle_rows(w, slice(0, 8))
    oracle.set_num_threads(1)
    try:
        rate1, rows1, dt1 = _oracle_rate(run1, 8, single_seconds)
    finally:
        oracle.set_num_threads(cores)
    return {"value": round(rate, 4), "unit": UNIT, "cores": cores, "kind": "oracle", "seconds": round(dt, 2),
            "sample": f"{rows} rows ({rows // batch_rows} x {batch_rows}) of the 8192x75968 bf16 workload, all four "
                      f"ops fwd+bwd, fp64 C oracle with OpenMP over rows; GB/s = the same algorithmic bytes per row "
                      f"as the GPU",
            "single_thread": {"value": round(rate1, 4), "unit": UNIT, "cores": 1, "seconds": round(dt1, 2),
                              "sample": f"{rows1} rows ({rows1 // 8} x 8), the same ops, one OpenMP thread"}}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    from vocab_wide_logprobs_gb300 import workloads
    oracle.build()
    rows = args.reference_rows
    w = workloads.pages_shape(seed=1, N=rows)
    run, _ = _oracle_rows(w, slice(0, rows))
    for _ in range(max(args.warmup, 3)):
        run()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run()
        times.append(time.perf_counter() - t0)
    dt = sum(times)
    step_bytes = sum(algorithmic_bytes(rows, VOCAB).values())
    value = step_bytes * args.steps / dt / 1e9
    line = {"metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": round(1e3 * dt / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD, "N": rows, "V": VOCAB, "note": f"bounded sample: {rows} rows per step"},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "kind": "oracle", "cores": oracle.num_threads(),
                             "sample": f"{rows} rows of the 8192x75968 bf16 workload per step, all four ops fwd+bwd"},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ---------------------------------------------------------------------------
# ranks
# ---------------------------------------------------------------------------
def _free_port() -> int:
    import socket
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def rank_command(n: int, argv, port: int) -> list:
    """torchrun command that starts n ranks of this script on one node (rendezvous on 127.0.0.1)."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
            "--master-addr", "127.0.0.1", f"--master-port={port}", os.path.abspath(__file__)] + list(argv)


def spawn_ranks(n: int, argv) -> int:
    """`--gpus n` without a launcher: start n ranks of this script, one per GPU, and return their
    exit status. Each rank times its own batch (rows are independent: replicas with no data-path
    collective); NCCL's initialisation log goes to stderr so that the rank count can be checked."""
    env = dict(os.environ)
    env.setdefault("NCCL_DEBUG", "INFO")
    env.setdefault("NCCL_DEBUG_SUBSYS", "INIT")
    env.setdefault("NCCL_DEBUG_FILE", "/dev/stderr")
    env.setdefault("OMP_NUM_THREADS", "1")
    return subprocess.call(rank_command(n, argv, _free_port()), env=env, cwd=ROOT)


def launch_check(rank: int, world: int, local_rank: int):
    """Rank plumbing without GPU work: every rank joins the process group (NCCL on GPUs, gloo
    otherwise), the max over ranks is taken as for a timing, and rank 0 prints who took part."""
    import torch
    import torch.distributed as dist
    cuda = torch.cuda.is_available()
    dev = torch.device("cuda", local_rank) if cuda else torch.device("cpu")
    if world > 1:
        if cuda:
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl", device_id=dev)
        else:
            dist.init_process_group("gloo")
    ranks = torch.zeros(world, dtype=torch.float64, device=dev)
    ranks[rank] = 1.0
    if world > 1:
        dist.all_reduce(ranks)
    slowest = max_over_ranks(float(rank + 1), dist if world > 1 else None, dev)
    if rank == 0:
        print(json.dumps({"launch_check": True, "n_gpus": world, "ranks_seen": int(ranks.sum().item()),
                          "max_over_ranks": slowest, "backend": (dist.get_backend() if world > 1 else None)}))
    if world > 1:
        dist.destroy_process_group()


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-strided", action="store_true", help="skip the strided and fp32-stress lines")
    p.add_argument("--reference-rows", type=int, default=64)
    p.add_argument("--rows", type=int, default=N_ROWS, help="rows per GPU (8192 is the benchmarked workload)")
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end measurement")
    p.add_argument("--no-linear", action="store_true", help="skip the fused linear-logp measurement")
    p.add_argument("--linear-only", action="store_true",
                   help="only the fused linear-logp measurement (profiling of the GEMM kernels)")
    p.add_argument("--linear-rows", type=int, default=8192, help="hidden rows of the linear-logp workload")
    p.add_argument("--linear-ops", default=None,
                   help="comma-separated op families of the linear line (logp, entropy, kl, jsd); default all")
    p.add_argument("--no-sustained", action="store_true", help="skip the linear line's sustained figures")
    p.add_argument("--launch-check", action="store_true",
                   help="only start the ranks, take the max over them and print who took part (no GPU work)")
    args = p.parse_args()
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        sys.exit(spawn_ranks(args.gpus, sys.argv[1:]))
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if args.gpus != world:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; launch one rank per GPU", file=sys.stderr)
        sys.exit(2)
    if args.launch_check:
        launch_check(rank, world, local_rank)
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
