"""Host logic of bench.py (no GPU): the algorithmic bytes behind its GB/s, the
clock summary that accepts or rejects a run, and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_algorithmic_bytes_of_the_step():
    N, V = 8192, 75968
    E = N * V * 2
    b = bench.algorithmic_bytes(N, V)
    assert sum(b.values()) == 18 * E                     # 22.40 GB per step at bf16
    assert b["logprobs_fwd"] == E and b["logprobs_bwd"] == 2 * E
    assert b["kl_rev_fwd"] == 2 * E and b["kl_fwd_bwd"] == 4 * E   # read A and B; write dA and dB too
    assert sum(bench.algorithmic_bytes(N, V, s=4).values()) == 2 * sum(b.values())


def test_clock_summary_takes_loaded_samples_and_throttle_reasons():
    c = bench.ClockSampler(0)
    c.proc = object()                                   # as if nvidia-smi had run
    rows = ["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 2070, 2070, 910.0, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 345, 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active",   # idle: left out
            "0, 1980, 2070, 1200.0, 0x4, Not Active, Not Active, Not Active, Active",
            "garbled line"]
    c.tmp.write("\n".join(rows) + "\n")
    c.tmp.flush()
    s = c.summary()
    os.unlink(c.tmp.name)
    assert s["sm_max_mhz"] == 2070.0 and s["sm_mhz"] == 2070.0 and s["samples"] == 4
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_reports_a_thermal_slowdown():
    c = bench.ClockSampler(0)
    c.proc = object()
    c.tmp.write("0, 1500, 2070, 1300.0, 0x40, Not Active, Active, Not Active, Not Active\n")
    c.tmp.flush()
    s = c.summary()
    os.unlink(c.tmp.name)
    assert s["reasons"] == ["hw_thermal_slowdown"] and s["sm_mhz"] == 1500.0


def test_reference_arm_prints_the_contract_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3",
                          "--reference-rows", "2"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["n_gpus"] == 1 and line["steps"] == 1 and line["warmup"] == 3 and line["higher_is_better"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["e2e"]["value"] == line["value"] == line["cpu_baseline"]["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["metric"] == bench.METRIC


def _max_rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 3.0 + rank * 0.5                           # rank 1 is the slower one
        worst = bench.max_over_ranks(ms, dist, "cpu")
        q.put((rank, worst, bench.job_rate_gbs(22.4e9, world, worst)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time_and_the_job_rate():
    """The N > 1 timing path of bench.py over gloo: every rank takes the max of the ranks'
    times, and the whole-job rate counts both ranks' bytes over that time."""
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_max_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict((r, (w, g)) for r, w, g in (q.get(timeout=150) for _ in procs))
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for r in range(2):
        assert res[r][0] == 3.5
        assert abs(res[r][1] - 2 * 22.4e9 / 3.5e-3 / 1e9) < 1e-9
    assert bench.max_over_ranks(1.25, None, "cpu") == 1.25


def test_gpus_two_starts_two_ranks_by_itself():
    """`bench.py --gpus 2` with no launcher starts two ranks (gloo without a GPU) and prints one line."""
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    out = subprocess.run([sys.executable, "bench.py", "--gpus", "2", "--launch-check"], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.strip().splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    line = json.loads(lines[0])
    assert line["n_gpus"] == 2 and line["ranks_seen"] == 2 and line["max_over_ranks"] == 2.0


def test_rank_command_uses_the_loopback_rendezvous():
    cmd = bench.rank_command(4, ["--steps", "3"], 29500)
    assert "--nproc-per-node=4" in cmd and "127.0.0.1" in cmd and cmd[-2:] == ["--steps", "3"]


def test_gpus_must_match_the_launcher():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    out = subprocess.run([sys.executable, "bench.py", "--gpus", "2", "--launch-check"], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=300)
    assert out.returncode == 2 and "WORLD_SIZE" in out.stderr


def test_ops_table_against_the_nominal_and_measured_peaks():
    # SURVEY-style table: fwd + bwd of each op, its bytes, the fraction of 8 TB/s and the 85% mark
    nbytes = bench.algorithmic_bytes(8192, 75968)
    per_op = {"logprobs_fwd": 0.2, "logprobs_bwd": 0.35, "entropy_fwd": 0.21, "entropy_bwd": 0.35,
              "kl_rev_fwd": 0.41, "kl_rev_bwd": 0.71, "kl_fwd_fwd": 0.41, "kl_fwd_bwd": 0.71}
    t = bench.ops_table(per_op, nbytes, {"hbm_gbs": 6775.6}, kl_da_only_ms=0.93)
    E2 = 8192 * 75968 * 2
    assert t["logprobs"]["bytes"] == 3 * E2 and t["kl_da_db"]["bytes"] == 6 * E2 and t["kl_da_only"]["bytes"] == 5 * E2
    assert abs(t["logprobs"]["ms"] - 0.55) < 1e-9
    assert abs(t["logprobs"]["mark_85pct_of_8tbps_ms"] - 3 * E2 / (0.85 * 8e12) * 1e3) < 1e-4   # 0.549 ms
    assert abs(t["kl_da_only"]["mark_85pct_of_8tbps_ms"] - 0.915) < 1e-3
    assert abs(t["kl_da_db"]["frac_of_8tbps"] - 6 * E2 / 1.12e-3 / 8e12) < 1e-4
