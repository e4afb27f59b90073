"""Host logic of bench.py: rank aggregation over gloo, clock parsing, reference arm."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    group = bench.init_group(world, "gloo")
    bench.barrier(group)
    mx = bench.reduce_over_ranks(group, 1.0 + rank, "max")
    sm = bench.reduce_over_ranks(group, 10.0 * (rank + 1), "sum")
    q.put((rank, mx, sm))
    group.destroy_process_group()


def test_replica_aggregation_gloo_two_ranks():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    # the slowest rank sets the time; units add up over ranks
    assert got == [(0, 2.0, 30.0), (1, 2.0, 30.0)]


def test_single_rank_aggregation_is_identity():
    assert bench.reduce_over_ranks(None, 3.5, "max") == 3.5
    assert bench.init_group(1, "gloo") is None


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3", "--workload", "tiny"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "GB/s" and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] == 1
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
    assert rec["metric"] == bench.METRIC


def test_reference_arm_bounds_its_sample():
    args = bench.parse_args(["--impl", "reference", "--steps", "50", "--warmup", "3",
                             "--reference-seconds", "0.05", "--workload", "attn"])
    rec = bench.run_reference(args, 0, 1)
    assert "first" in rec["cpu_baseline"]["sample"]
    assert int(rec["cpu_baseline"]["sample"].split()[1]) < 4096


def test_clock_parsing():
    text = "\n".join([
        "0, 1965, 2070, 812.3, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 900.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1950, 2070, 850.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ])
    c = bench.parse_clock_samples(text)
    assert c["sm_mhz"] == 1965 and c["sm_max_mhz"] == 2070 and c["samples"] == 3
    assert c["reasons"] == ["sw_power_cap"]
    assert bench.parse_clock_samples("") is None


def test_traffic_ignored_when_kernel_changed(tmp_path, monkeypatch):
    rec = {"workloads": {
        "attn": {"dram_bytes_per_launch": 123, "kernel_source": "regs_kernel.cuh",
                 "kernel_source_sha256": "0" * 64},
        "attn_m4_regs": {"dram_bytes_per_launch": 456, "kernel_source": "batched.cuh",
                    "kernel_source_sha256": bench.kernel_source_hash("batched.cuh")},
        "tiny": {"dram_bytes_per_launch": 789, "kernel_source": "no_such_file.cuh",
                 "kernel_source_sha256": "0" * 64}}}
    p = tmp_path / "traffic.json"
    p.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(p))
    assert bench.recorded_traffic("attn") is None  # the kernel changed since the capture
    assert bench.recorded_traffic(bench.traffic_key("attn", 4, kernel=1)) == 456
    assert bench.recorded_traffic(bench.traffic_key("attn", 4, kernel=7)) is None  # another kernel's capture
    assert bench.recorded_traffic("tiny") is None
    assert bench.recorded_traffic("ffn_up") is None
    rec["workloads"]["attn"]["kernel_source_sha256"] = bench.kernel_source_hash("regs_kernel.cuh")
    p.write_text(json.dumps(rec))
    assert bench.recorded_traffic(bench.traffic_key("attn", 1)) == 123


def test_tc_calls_count_two_launches():
    assert bench.launches_per_call({"kernel": 7}) == 2
    assert bench.launches_per_call({"kernel": 1}) == 1
    assert bench.traffic_key("up70b", 16, kernel=7) == "up70b_m16_tc"


def test_bench_rejects_short_warmup():
    with pytest.raises(SystemExit):
        bench.parse_args(["--warmup", "2"])


def test_all_core_oracle_baseline_runs_one_process_per_core():
    import workloads

    wl = workloads.WORKLOADS["tiny"]
    A, W, S = workloads.make_inputs(wl)
    rec = bench.cpu_all_cores(A, W, S, wl, 1, 0.2)
    assert rec["cores"] == min(len(bench.affinity_cores()), wl.N)
    assert rec["value"] > 0 and rec["unit"] == "GB/s"
    full = bench.cpu_baseline(A, W, S, wl.algorithmic_bytes(), 0.2, wl, all_core_seconds=0.2)
    assert full["kind"] == "oracle" and full["cpu_model"]
    assert full["single_thread"]["cores"] == 1
    assert full["cores"] == rec["cores"]
