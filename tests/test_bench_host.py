"""Host-side pieces of bench.py, without a GPU: the multi-rank timing
reduction over gloo (world size 2), clock-sample parsing, and the reference
arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), TQ_BENCH_BACKEND="gloo")
    sys.path.insert(0, ROOT)
    import bench
    r, w, _ = bench.dist_init(world)
    bench.barrier(w)
    got = bench.max_over_ranks(1.5 + r, w)
    out_q.put((r, w, got))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert res == [(0, 2, 2.5), (1, 2, 2.5)]


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_clock_summary_parsing():
    sys.path.insert(0, ROOT)
    import bench
    c = bench.ClockSampler(0)
    c.lines = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1965, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1201.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    s = c.summary()
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    empty = bench.ClockSampler(0)
    assert empty.summary()["samples"] == 0


def test_algorithmic_bytes_of_the_decode_workload():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.algorithmic_bytes(32768, 8192, 1) == 71303168 + 9344 + 131072


def test_reference_arm_prints_one_json_line():
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "0"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert p.returncode == 0, p.stderr
    lines = [ln for ln in p.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "Gweights/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    sys.path.insert(0, ROOT)
    import bench
    assert d["metric"] == bench.metric_name("Gweights/s", "decode")   # the GPU arm's string


def test_graph_plan_times_exactly_the_requested_steps():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.graph_plan(20000, 5) == (40, 500, 0)     # decode: 5 weight copies
    assert bench.graph_plan(2002, 13) == (39, 51, 13)     # 13 copies of a 24 MB matrix
    assert bench.graph_plan(20, 5) == (40, 0, 20)         # fewer steps than one graph
    assert bench.graph_plan(7, 64) == (64, 0, 7)          # more copies than the graph size
    for steps in range(1, 300, 7):
        for copies in (2, 5, 13, 41, 64):
            G, reps, rest = bench.graph_plan(steps, copies)
            assert G % copies == 0 and G >= copies and 0 <= rest < G
            assert reps * G + rest == steps


def test_e2e_streams_option():
    sys.path.insert(0, ROOT)
    import bench
    argv = sys.argv
    try:
        sys.argv = ["bench.py"]
        assert bench.parse_args().e2e_streams == 4
        sys.argv = ["bench.py", "--e2e-streams", "2"]
        assert bench.parse_args().e2e_streams == 2
    finally:
        sys.argv = argv


def test_source_hash_ignores_comments():
    sys.path.insert(0, ROOT)
    import bench
    a = "int f(int x) {  // one\n  return x; /* two\n lines */ }\n"
    b = "int f(int x) {  // other words\n  return x; /* x */ }\n"
    c = "int f(int x) {\n  return x + 1; }\n"
    assert bench.code_text(a) == bench.code_text(b)
    assert bench.code_text(a) != bench.code_text(c)
    assert "return x;" in bench.code_text(a) and "one" not in bench.code_text(a)
    # a comment line added or removed changes nothing either
    assert bench.code_text("int f();\n// added\nint g();\n") == bench.code_text("int f();\nint g();\n")


def test_launch_count_follows_the_staging_rule():
    """gpu_launches counts what tq_quantize_matmul enqueues: one fused GEMV, or
    from 4 tokens where the workspace size is not 0 (3072 columns and more) a
    staging kernel and the GEMV, and two launches on the tensor-core path."""
    sys.path.insert(0, ROOT)
    import bench
    from bit_matvec_gb300 import build
    build.build()
    assert bench.launches_per_matmul(32768, 8192, 1) == 1
    assert bench.launches_per_matmul(17408, 5120, 3) == 1
    assert bench.launches_per_matmul(17408, 5120, 4) == 2
    assert bench.launches_per_matmul(17408, 2048, 4) == 1
    assert bench.launches_per_matmul(17408, 5120, 64) == 2
    assert bench.gemv_kernel_name(17408, 5120, 4).startswith("gemv_stage_kernel")
    assert bench.gemv_kernel_name(32768, 8192, 1).startswith("gemv_kernel")
